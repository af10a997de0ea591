// fa_fwd_f32x3.cu -- fp32 attention forward on the sm_103a tensor cores.
//
// The `Float32` interface of `mo.mha.no_cache` (MAX API page
// "FlashAttentionGPU": scale is Float32, tensors may be fp32) at fp32
// accuracy, without the CUDA-core kernel's FMA rate. Every fp32 operand x is
// split into three bf16 parts, x = b0 + b1 + b2 + r with |r| <= 2^-24 |x|
// (b0 = bf16(x), b1 = bf16(x - b0), b2 = bf16(x - b0 - b1); both
// subtractions are exact in fp32). A product x y is then the sum of the six
// part products whose size is at least 2^-16 of b0 b0:
//   b0b0 + b0b1 + b1b0 + b1b1 + b0b2 + b2b0,
// each a bf16 tcgen05.mma with fp32 accumulation; the dropped terms are
// about 2^-23 relative. Both contractions of the FlashAttention-2 loop
// (tiny_flash_attn.py page, flash_attn_v2) use this:
//   S = Q K^T  from Q's parts in tensor memory (A operand) and K's parts in
//              shared memory (split once per call into bf16 planes by
//              split_planes_kernel, then streamed by TMA like the bf16 path);
//   O += P V   from P's parts in tensor memory and V's parts in shared memory.
// Softmax, masking and the lazy O rescale are those of the bf16 kernel, in
// fp32, on 64-key tiles.
//
// Tensor memory (D = 128; 512 columns): Q parts at 0, 64, 128 (bf16 pairs),
// S double-buffered at 192 and 256 (P0 written over the first 32 columns of
// its S buffer), P1 at 320, P2 at 352, O at 384. D = 64 uses half the Q and O
// columns.
//
// Warp roles (192 threads): warps 0-3 softmax (thread = query row = lane),
// warp 4 MMA issuer, warp 5 TMA producer. Every mbarrier wait is bounded.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;                 // query rows per CTA (= TMEM lanes)
constexpr int kBN = 64;                  // keys per K/V tile
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kBoxBytes = kBN * 128;     // [64 rows][64 bf16], 128B-swizzled
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr unsigned long long kDrainExtraNs = 100000000ull;
constexpr uint32_t kNegInfBits = 0xff800000u;

// The six (i, j) part pairs of a product, largest first.
__device__ constexpr int kPairA[6] = {0, 0, 1, 1, 0, 2};
__device__ constexpr int kPairB[6] = {0, 1, 0, 1, 2, 0};

template <int D>
struct X3Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kPartBytes = (D / 64) * kBoxBytes;  // one part of a [64][D] tile
  static constexpr int kSlotBytes = 3 * kPartBytes;         // K or V tile, three parts
  static constexpr int kStages = D == 128 ? 4 : 8;
  static constexpr int kKVOff = 0;
  static constexpr int kBarOff = kKVOff + kStages * kSlotBytes;
  // q_ready kv_full[S] kv_empty[S] s_full[2] p_full[2] pv_done o_full drain
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  // Tensor-memory columns.
  static constexpr uint32_t kColQ = 0;            // part p at kColQ + p * D / 2
  static constexpr uint32_t kColS = 3 * D / 2;    // buffer t at kColS + 64 t
  static constexpr uint32_t kColP1 = kColS + 128;
  static constexpr uint32_t kColP2 = kColP1 + 32;
  static constexpr uint32_t kColO = kColP2 + 32;
  static_assert(kColO + D <= kTmemCols, "tensor memory");
};

// Three bf16 parts of x (bit patterns in the low 16 bits).
__device__ __forceinline__ void split3(float x, uint32_t& h0, uint32_t& h1, uint32_t& h2) {
  const __nv_bfloat16 a = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(a);
  const __nv_bfloat16 b = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(b);
  const __nv_bfloat16 c = __float2bfloat16_rn(r2);
  h0 = __bfloat16_as_ushort(a);
  h1 = __bfloat16_as_ushort(b);
  h2 = __bfloat16_as_ushort(c);
}

__global__ void __launch_bounds__(256)
    split_planes_kernel(const float* __restrict__ src, long long n, uint16_t* __restrict__ p0,
                        uint16_t* __restrict__ p1, uint16_t* __restrict__ p2) {
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n; i += 256ll * gridDim.x) {
    uint32_t a, b, c;
    split3(src[i], a, b, c);
    p0[i] = static_cast<uint16_t>(a);
    p1[i] = static_cast<uint16_t>(b);
    p2[i] = static_cast<uint16_t>(c);
  }
}

// Hides (-inf) scores outside the visible columns [vlo, vhi] of a 64-key
// tile; with a zero scale the visible ones become 0.
__device__ __forceinline__ void mask_cols64(uint32_t* r, int vlo, int vhi, bool zero_scale) {
  int lo = max(vlo, 0);
  const int hi = min(vhi, kBN - 1);
  unsigned span = static_cast<unsigned>(hi - lo);
  if (hi < lo) {
    lo = 2 * kBN;
    span = 0;
  }
  const uint32_t keep = zero_scale ? 0u : 0xffffffffu;
#pragma unroll
  for (int e = 0; e < kBN; ++e)
    r[e] = static_cast<unsigned>(e - lo) <= span ? (r[e] & keep) : kNegInfBits;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_f32x3_kernel(const __grid_constant__ CUtensorMap tk0,
                        const __grid_constant__ CUtensorMap tk1,
                        const __grid_constant__ CUtensorMap tk2,
                        const __grid_constant__ CUtensorMap tv0,
                        const __grid_constant__ CUtensorMap tv1,
                        const __grid_constant__ CUtensorMap tv2, const F32x3Problem p,
                        int num_qblocks) {
  using C = X3Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sKV = base + C::kKVOff;
  const uint32_t bars = base + C::kBarOff;
  const uint32_t bar_q_ready = bars;
  const uint32_t bar_kv_full = bars + 8;
  const uint32_t bar_kv_empty = bars + 8 * (1 + C::kStages);
  const uint32_t bar_s_full = bars + 8 * (1 + 2 * C::kStages);
  const uint32_t bar_p_full = bar_s_full + 16;
  const uint32_t bar_pv_done = bar_p_full + 16;
  const uint32_t bar_o_full = bar_pv_done + 8;
  const uint32_t bar_drain = bar_o_full + 8;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: the CTAs of one (batch, KV head) -- every query block of each
  // of its G query heads -- are consecutive, heaviest (last) query blocks
  // first, so the K/V planes they all stream stay in L2 while they run
  // (query block major, the planes were read from DRAM again by each wave).
  const int G = p.H / p.Hkv;
  const int per_group = num_qblocks * G;
  const int grp = static_cast<int>(blockIdx.x / per_group);
  const int rem = static_cast<int>(blockIdx.x % per_group);
  const int qb = num_qblocks - 1 - rem / G;
  const int hk = grp % p.Hkv;
  const int b = grp / p.Hkv;
  const int h = hk * G + rem % G;
  const int q0 = qb * kBM;
  const int kv_end = p.causal ? min(p.S, q0 + kBM)
                              : (p.window > 0 ? min(p.S, q0 + kBM - 1 + p.window) : p.S);
  const int kv_begin = p.window > 0 ? max(0, q0 - p.window + 1) : 0;
  const int jlo = kv_begin / kBN;
  const int jhi = (kv_end + kBN - 1) / kBN;
  const int n = jhi - jlo;
  const unsigned long long limit = p.wait_limit_ns;
  const unsigned long long drain_limit = limit + kDrainExtraNs;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_q_ready, 4);
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar_kv_full + 8 * s, 1);
      ptx::mbar_init(bar_kv_empty + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar_s_full + 8 * t, 1);
      ptx::mbar_init(bar_p_full + 8 * t, 4);
    }
    ptx::mbar_init(bar_pv_done, 1);
    ptx::mbar_init(bar_o_full, 1);
    ptx::mbar_init(bar_drain, 1);
    misc[1] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::tma_prefetch_desc(&tk0);
    ptx::tma_prefetch_desc(&tk1);
    ptx::tma_prefetch_desc(&tk2);
    ptx::tma_prefetch_desc(&tv0);
    ptx::tma_prefetch_desc(&tv1);
    ptx::tma_prefetch_desc(&tv2);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(base + C::kMiscOff, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];

  auto fail = [&]() {
    misc[1] = 1;
    atomicOr(p.status, kStatusWaitTimeout);
  };
  auto aborted = [&]() { return misc[1] != 0; };

  if (warp == kLoadWarp) {
    // ===================================================== TMA producer
    if (lane == 0 && n > 0) {
      const uint64_t pol = ptx::policy_evict_last();
      uint32_t armed = 0, armed_parity = 0;
      int idx = 0;
      bool ok = true;
      auto issue = [&](int kind, int j) {
        const int s = idx % C::kStages;
        const uint32_t ph = static_cast<uint32_t>(idx / C::kStages) & 1u;
        ++idx;
        if (aborted() || !ptx::mbar_wait(bar_kv_empty + 8 * s, ph ^ 1u, limit)) {
          fail();
          ok = false;
          return;
        }
        ptx::mbar_arrive_expect_tx(bar_kv_full + 8 * s, C::kSlotBytes);
        const CUtensorMap* m0 = kind == 0 ? &tk0 : &tv0;
        const CUtensorMap* m1 = kind == 0 ? &tk1 : &tv1;
        const CUtensorMap* m2 = kind == 0 ? &tk2 : &tv2;
        const uint32_t dst = sKV + s * C::kSlotBytes;
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) {
          ptx::tma_load_4d(dst + bx * kBoxBytes, m0, bar_kv_full + 8 * s, bx * 64, hk, j * kBN, b,
                           pol);
          ptx::tma_load_4d(dst + C::kPartBytes + bx * kBoxBytes, m1, bar_kv_full + 8 * s,
                           bx * 64, hk, j * kBN, b, pol);
          ptx::tma_load_4d(dst + 2 * C::kPartBytes + bx * kBoxBytes, m2, bar_kv_full + 8 * s,
                           bx * 64, hk, j * kBN, b, pol);
        }
        armed |= 1u << s;
        armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
      };
      // Ring order = MMA consumption order: K0 K1 | V0 K2 | V1 K3 | ...
      issue(0, jlo);
      if (ok && n > 1) issue(0, jlo + 1);
      for (int r = 0; r < n && ok; ++r) {
        issue(1, jlo + r);
        if (ok && r + 2 < n) issue(0, jlo + r + 2);
      }
      for (int s = 0; s < C::kStages; ++s)
        if ((armed >> s) & 1u)
          ptx::mbar_wait(bar_kv_full + 8 * s, (armed_parity >> s) & 1u, drain_limit);
    }
  } else if (warp == kMmaWarp) {
    // ===================================================== MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, D, false, true);
      bool ok = true;
      if (p.stall_probe && !ptx::mbar_wait(bar_drain, 0, limit)) {
        fail();
        ok = false;
      }
      if (ok && !ptx::mbar_wait(bar_q_ready, 0, limit)) {
        fail();
        ok = false;
      }
      ptx::tc_fence_after();
      int idx = 0;
      auto wait_kv = [&]() -> int {
        const int s = idx % C::kStages;
        const uint32_t ph = static_cast<uint32_t>(idx / C::kStages) & 1u;
        ++idx;
        if (aborted() || !ptx::mbar_wait(bar_kv_full + 8 * s, ph, limit)) {
          fail();
          return -1;
        }
        ptx::tc_fence_after();
        return s;
      };
      const uint64_t dk0 = ptx::smem_desc_sw128(sKV, 16, 1024);
      const uint64_t dv0 = ptx::smem_desc_sw128(sKV, kBoxBytes, 1024);
      auto issue_s = [&](int buf, int kslot) {
        const uint32_t d_s = tmem + C::kColS + 64 * buf;
#pragma unroll
        for (int pr = 0; pr < 6; ++pr) {
          const uint32_t a_q = tmem + C::kColQ + kPairA[pr] * (D / 2);
          const uint64_t dk = dk0 + static_cast<uint32_t>(
                                        (kslot * C::kSlotBytes + kPairB[pr] * C::kPartBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off =
                static_cast<uint32_t>(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
            ptx::mma_ts(d_s, a_q + kk * 8, dk + off, kIdescS, (pr > 0 || kk > 0) ? 1u : 0u);
          }
        }
        ptx::tc_commit(bar_s_full + 8 * buf);
        ptx::tc_commit(bar_kv_empty + 8 * kslot);
      };
      auto issue_pv = [&](int buf, int vslot, bool accumulate) {
        const uint32_t a_p[3] = {tmem + C::kColS + 64 * buf, tmem + C::kColP1, tmem + C::kColP2};
#pragma unroll
        for (int pr = 0; pr < 6; ++pr) {
          const uint64_t dv = dv0 + static_cast<uint32_t>(
                                        (vslot * C::kSlotBytes + kPairB[pr] * C::kPartBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            ptx::mma_ts(tmem + C::kColO, a_p[kPairA[pr]] + kk * 8,
                        dv + static_cast<uint32_t>(kk * 128), kIdescPV,
                        (accumulate || pr > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::tc_commit(bar_pv_done);
        ptx::tc_commit(bar_kv_empty + 8 * vslot);
      };

      if (ok) {
        const int ks = wait_kv();
        if (ks < 0) ok = false;
        else issue_s(0, ks);
      }
      if (ok && n > 1) {
        const int ks = wait_kv();
        if (ks < 0) ok = false;
        else issue_s(1, ks);
      }
      for (int r = 0; ok && r < n; ++r) {
        const int buf = r & 1;
        const int vs = wait_kv();
        if (vs < 0) break;
        if (aborted() || !ptx::mbar_wait(bar_p_full + 8 * buf, (r >> 1) & 1, limit)) {
          fail();
          break;
        }
        ptx::tc_fence_after();
        issue_pv(buf, vs, r > 0);
        if (r + 2 < n) {
          const int ks = wait_kv();
          if (ks < 0) break;
          issue_s(buf, ks);
        }
      }
      ptx::tc_commit(bar_o_full);
      ptx::tc_commit(bar_drain);
      ptx::mbar_wait(bar_drain, 0, drain_limit);
    }
    __syncwarp();
  } else {
    // ===================================================== softmax warps
    const int quad = warp;
    const int row = quad * 32 + lane;
    const int i = q0 + row;
    const bool valid = i < p.S;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tO = tmem + lane_base + C::kColO;

    // Q row -> three bf16 parts -> tensor memory (64 columns per store).
    {
      const float* qrow = p.q + (static_cast<size_t>(b) * p.sq.b + static_cast<size_t>(i) * p.sq.s +
                                 static_cast<size_t>(h) * p.sq.h);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 64) {
        uint32_t part[3][32];
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (valid) v = *reinterpret_cast<const float4*>(qrow + c0 + e);
          uint32_t a0, a1, a2, b0, b1, b2, c0b, c1b, c2b, d0, d1, d2;
          split3(v.x, a0, a1, a2);
          split3(v.y, b0, b1, b2);
          split3(v.z, c0b, c1b, c2b);
          split3(v.w, d0, d1, d2);
          part[0][e / 2] = a0 | (b0 << 16);
          part[1][e / 2] = a1 | (b1 << 16);
          part[2][e / 2] = a2 | (b2 << 16);
          part[0][e / 2 + 1] = c0b | (d0 << 16);
          part[1][e / 2 + 1] = c1b | (d1 << 16);
          part[2][e / 2 + 1] = c2b | (d2 << 16);
        }
#pragma unroll
        for (int pp = 0; pp < 3; ++pp)
          ptx::tmem_st_32x32b_x32(tmem + lane_base + C::kColQ + pp * (D / 2) + c0 / 2, part[pp]);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_q_ready);
    }

    const int vlo = p.window > 0 ? i - p.window + 1 : INT_MIN;
    const int vhi = p.causal ? min(i, p.S - 1)
                             : (p.window > 0 ? min(i + p.window - 1, p.S - 1) : p.S - 1);
    const float c = p.scale_log2;
    const bool zero_scale = !(c > 0.f);
    const float ce = zero_scale ? 1.f : c;
    float m_use = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int r = 0; r < n; ++r) {
      const int buf = r & 1;
      const uint32_t tS = tmem + lane_base + C::kColS + 64 * buf;
      bool w = ptx::mbar_wait(bar_s_full + 8 * buf, (r >> 1) & 1, limit);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        fail();
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t s[kBN];
      float pm[2];  // maximum of each 32 columns, reduced by the load
      ptx::tmem_ld_max_32x32b_x32(tS, s, &pm[0]);
      ptx::tmem_ld_max_32x32b_x32(tS + 32, s + 32, &pm[1]);
      ptx::tmem_wait_ld();
      ptx::reg_fence<kBN>(s);
      asm volatile("" : "+f"(pm[0]), "+f"(pm[1]));  // no use above the wait

      const int k0 = (jlo + r) * kBN;
      bool full = k0 + kBN <= p.S;
      if (p.causal) full = full && (k0 + kBN - 1 <= q0);
      if (p.window > 0) full = full && (q0 + kBM - 1 - k0 < p.window);
      if (p.window > 0 && !p.causal) full = full && (k0 + kBN - 1 - q0 < p.window);
      if (!full || zero_scale)
        mask_cols64(s, vlo == INT_MIN ? INT_MIN : vlo - k0, vhi - k0, zero_scale);

      // Row maximum: from the loads' reductions when no score is hidden.
      float mx = -INFINITY;
      if (full && !zero_scale) {
        mx = fmaxf(pm[0], pm[1]);
      } else {
#pragma unroll
        for (int e = 0; e < kBN; e += 2)
          mx = ptx::max3(mx, __uint_as_float(s[e]), __uint_as_float(s[e + 1]));
      }
      const float m_tile = mx == -INFINITY ? -INFINITY : mx * ce;
      const float m_new = fmaxf(m_use, m_tile);
      float alpha = 1.f;
      bool rescale = false;
      if (r == 0) {
        m_use = m_new;
      } else if (m_new > m_use + kRescaleThreshold) {
        alpha = ptx::ex2_approx(m_use - m_new);
        m_use = m_new;
        rescale = true;
      }
      const float neg_base = m_use == -INFINITY ? 0.f : -m_use;
      // P in fp32, its row sum, and its three bf16 parts (pairs).
      uint32_t p0[kBN / 2], p1[kBN / 2], p2[kBN / 2];
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int e = 0; e < kBN; e += 2) {
        const float pa = ptx::ex2_approx(fmaf(__uint_as_float(s[e]), ce, neg_base));
        const float pb = ptx::ex2_approx(fmaf(__uint_as_float(s[e + 1]), ce, neg_base));
        sum0 += pa;
        sum1 += pb;
        uint32_t a0, a1, a2, b0, b1, b2;
        split3(pa, a0, a1, a2);
        split3(pb, b0, b1, b2);
        p0[e / 2] = a0 | (b0 << 16);
        p1[e / 2] = a1 | (b1 << 16);
        p2[e / 2] = a2 | (b2 << 16);
      }
      l_run = l_run * alpha + (sum0 + sum1);
      ptx::tmem_st_32x32b_x32(tS, p0);  // P0 over the first 32 columns of S
      // P1 and P2 are single-buffered: PV(r - 1) must have read them (and
      // have updated O, if it is rescaled) before they are overwritten.
      if (r > 0) {
        bool wp = ptx::mbar_wait(bar_pv_done, (r - 1) & 1, limit);
        wp = __all_sync(0xffffffffu, wp);
        if (!wp) {
          fail();
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      ptx::tmem_st_32x32b_x32(tmem + lane_base + C::kColP1, p1);
      ptx::tmem_st_32x32b_x32(tmem + lane_base + C::kColP2, p2);
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          ptx::tmem_ld_32x32b_x32(tO + c0, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence<32>(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          ptx::tmem_st_32x32b_x32(tO + c0, o);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full + 8 * buf);
    }

    // ---- epilogue: O / l (fp32) straight to global; LSE.
    if (ok && n > 0) {
      bool w = ptx::mbar_wait(bar_o_full, 0, limit);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        fail();
        ok = false;
      }
      ptx::tc_fence_after();
    }
    if (ok && n > 0) {
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      float* orow = p.out + (static_cast<size_t>(b) * p.so.b + static_cast<size_t>(i) * p.so.s +
                             static_cast<size_t>(h) * p.so.h);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        ptx::tmem_ld_32x32b_x32(tO + c0, o);
        ptx::tmem_wait_ld();
        ptx::reg_fence<32>(o);
        if (valid) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(orow + c0 + 4 * u) = make_float4(
                __uint_as_float(o[4 * u]) * inv_l, __uint_as_float(o[4 * u + 1]) * inv_l,
                __uint_as_float(o[4 * u + 2]) * inv_l, __uint_as_float(o[4 * u + 3]) * inv_l);
        }
      }
      if (valid && p.lse != nullptr) {
        const float m_fin = m_use == -INFINITY ? 0.f : m_use;
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.S + i] = (m_fin + __log2f(l_run)) * kLn2;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

bool encode_plane_map(CUtensorMap* m, const uint16_t* base, const F32x3Problem& p) {
  return encode_bshd_tensor_map(m, base, p.B, p.S, p.Hkv, p.D, BshdStrides{}, 1, kBN);
}

template <int D>
cudaError_t launch_d(const F32x3Problem& p, cudaStream_t stream) {
  // Split K and V into their bf16 planes (dense [B, S, Hkv, D] each).
  const long long nkv = static_cast<long long>(p.B) * p.S * p.Hkv * D;
  const long long sb = (nkv + 255) / 256;
  const int sblocks = static_cast<int>(sb < 152ll * 16 ? sb : 152ll * 16);
  split_planes_kernel<<<sblocks, 256, 0, stream>>>(p.k, nkv, p.kp[0], p.kp[1], p.kp[2]);
  split_planes_kernel<<<sblocks, 256, 0, stream>>>(p.v, nkv, p.vp[0], p.vp[1], p.vp[2]);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  CUtensorMap tk[3], tv[3];
  for (int t = 0; t < 3; ++t)
    if (!encode_plane_map(&tk[t], p.kp[t], p) || !encode_plane_map(&tv[t], p.vp[t], p))
      return cudaErrorInvalidValue;
  const int nqb = (p.S + kBM - 1) / kBM;
  const long long grid = static_cast<long long>(nqb) * p.H * p.B;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  static unsigned long long attr_done = 0;
  err = ensure_smem_attr(&attr_done, reinterpret_cast<const void*>(&fa_fwd_f32x3_kernel<D>),
                         X3Cfg<D>::kSmemBytes);
  if (err != cudaSuccess) return err;
  fa_fwd_f32x3_kernel<D><<<static_cast<unsigned>(grid), kThreads, X3Cfg<D>::kSmemBytes, stream>>>(
      tk[0], tk[1], tk[2], tv[0], tv[1], tv[2], p, nqb);
  return cudaGetLastError();
}

}  // namespace

unsigned long long f32x3_workspace_bytes(int B, int S, int Hkv, int D) {
  const unsigned long long plane = static_cast<unsigned long long>(B) * S * Hkv * D * 2ull;
  return 6ull * ((plane + 255ull) & ~255ull);
}

cudaError_t launch_fwd_f32x3_tc(F32x3Problem p, void* workspace, cudaStream_t stream) {
  const unsigned long long plane =
      (static_cast<unsigned long long>(p.B) * p.S * p.Hkv * p.D * 2ull + 255ull) & ~255ull;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  for (int t = 0; t < 3; ++t) {
    p.kp[t] = reinterpret_cast<uint16_t*>(w + t * plane);
    p.vp[t] = reinterpret_cast<uint16_t*>(w + (3 + t) * plane);
  }
  p.sq = resolve_strides(p.sq, p.S, p.H, p.D);
  p.so = resolve_strides(p.so, p.S, p.H, p.D);
  if (p.D == 64) return launch_d<64>(p, stream);
  if (p.D == 128) return launch_d<128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
