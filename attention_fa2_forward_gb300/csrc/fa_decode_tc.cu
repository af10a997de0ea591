// fa_decode_tc.cu -- bf16 attention over a KV cache on the sm_103a tensor
// cores: the cached sibling of `mo.mha.no_cache` (MAX API page
// "FlashAttentionGPU", method `execute`). Batch b holds L_b keys and values
// at the start of a cache of capacity S_cache ([B, S_cache, Hkv, D]); its Sq
// queries ([B, Sq, H, D]) are the last Sq tokens of the sequence, so query
// row s sits at position L_b - Sq + s and the mask is evaluated there. Keys
// at positions >= L_b are never used; a query that sees no key gets O = 0
// and LSE = -inf.
//
// Decoding reads the whole cache once per step and does little arithmetic
// per byte, so HBM bandwidth bounds it. The design keeps the FlashAttention-2
// loop of the prefill kernel (online softmax, O rescaled lazily, one final
// division) and changes the work decomposition:
//
//   * the G query heads that share one KV head, times Pq query positions
//     (Pq = min(Sq, 128 / G)), fill the 128 rows of one MMA tile, row
//     r = position * G + head; the Q tile is one TMA box {64, G, Pq} per
//     64 columns, so every K/V tile is read once for the whole group;
//   * a CTA owns one (split, KV head, position tile, batch) and streams its
//     share of the KV tiles through a 6-slot ring; when the (b, KV head)
//     units alone cannot fill the GPU, the key range is cut into splits
//     whose partial results (O / l in fp32 and the LSE) a second kernel
//     merges with weights exp(LSE_split - LSE);
//   * S is double-buffered in tensor memory (S_0, S_1 at columns 0 and 128,
//     O at 256): the MMA warp computes S(j+1) while the softmax warps work
//     on S(j). The issue order is S0 S1 | PV0 S2 | PV1 S3 | ...;
//   * only the softmax warps whose tensor-memory lanes hold real rows work;
//   * V rows of the last tile that lie past L_b but inside the cache are
//     zeroed in shared memory before the PV MMA reads them (their P is 0, but
//     0 * NaN would not be).
//
// Every mbarrier wait is bounded (global timer); on time-out the CTA records
// kStatusWaitTimeout, stops issuing work, waits (bounded) for its own copies
// and MMAs, releases tensor memory and returns.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "fa_internal.h"
#include "fa_tile.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;                 // rows per Q tile (= TMEM lanes)
constexpr int kBN = tile::kBN;           // keys per K/V tile
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kThreads = 6 * 32;         // 4 softmax warps, MMA warp, TMA warp
constexpr int kBoxBytes = kBN * 128;     // [128 rows][64 bf16], 128B-swizzled
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;          // O at columns [256, 256 + D)
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr unsigned long long kDrainExtraNs = 100000000ull;  // 100 ms

template <int D>
struct DCfg {
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  // Ring slots: what fits next to the Q tile in 227 KB. Two slots suffice for
  // the ring order (K0 K1 | V0 K2 | ...): each refill waits only on an MMA
  // that needs nothing later in the ring.
  static constexpr int kStages = D == 256 ? 2 : (D == 128 ? 6 : 10);
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // q_full kv_full[S] kv_empty[S] s_full[2] p_full[2] pv_done o_full v_fixed drain
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack for 1 KB alignment
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_decode_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                             const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ CUtensorMap tm_o, const DecodeProblem p) {
  using C = DCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kQOff;
  const uint32_t sKV = base + C::kKVOff;
  const uint32_t bars = base + C::kBarOff;
  const uint32_t bar_q_full = bars;
  const uint32_t bar_kv_full = bars + 8;                          // + 8 s
  const uint32_t bar_kv_empty = bars + 8 * (1 + C::kStages);      // + 8 s
  const uint32_t bar_s_full = bars + 8 * (1 + 2 * C::kStages);    // + 8 buf
  const uint32_t bar_p_full = bar_s_full + 16;                    // + 8 buf
  const uint32_t bar_pv_done = bar_p_full + 16;
  const uint32_t bar_o_full = bar_pv_done + 8;
  const uint32_t bar_v_fixed = bar_o_full + 8;
  const uint32_t bar_drain = bar_v_fixed + 8;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
  // misc[0]: tensor-memory base address, misc[1]: abort flag

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: split fastest, then KV head, position tile, batch
  unsigned id = blockIdx.x;
  const int split = static_cast<int>(id % static_cast<unsigned>(p.splits));
  id /= static_cast<unsigned>(p.splits);
  const int hk = static_cast<int>(id % static_cast<unsigned>(p.Hkv));
  id /= static_cast<unsigned>(p.Hkv);
  // Later position tiles see more keys under the causal mask: start them first.
  const int pt = p.n_ptiles - 1 - static_cast<int>(id % static_cast<unsigned>(p.n_ptiles));
  const int b = static_cast<int>(id / static_cast<unsigned>(p.n_ptiles));

  const int L = min(max(p.lens != nullptr ? p.lens[b] : p.Scache, 0), p.Scache);
  const int sq0 = pt * p.Pq;              // first query row of the tile
  const int nq = min(p.Pq, p.Sq - sq0);   // query positions in the tile
  const int pos0 = L - p.Sq + sq0;        // position of the first of them
  const int posl = pos0 + nq - 1;
  // Keys any row of the tile may see: [klo, khi].
  const int klo = p.window > 0 ? max(0, pos0 - p.window + 1) : 0;
  const int khi = p.causal ? min(posl, L - 1)
                           : (p.window > 0 ? min(posl + p.window - 1, L - 1) : L - 1);
  // This CTA's KV tiles [jlo, jhi).
  int jlo = 0, jhi = 0;
  if (khi >= klo) {
    const int t0 = klo / kBN, t1 = khi / kBN + 1;
    jlo = t0 + split * p.tiles_per_split;
    jhi = max(jlo, min(t1, jlo + p.tiles_per_split));
  }
  const int n = jhi - jlo;
  // The last tile holds cache rows past L_b: zero those V rows.
  const bool v_fix = n > 0 && (L % kBN) != 0 && L < p.Scache && jhi - 1 == L / kBN;
  const int nact = (p.R + 31) >> 5;       // softmax warps holding real rows
  const unsigned long long limit = p.wait_limit_ns;
  const unsigned long long drain_limit = limit + kDrainExtraNs;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar_kv_full + 8 * s, 1);
      ptx::mbar_init(bar_kv_empty + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar_s_full + 8 * t, 1);
      ptx::mbar_init(bar_p_full + 8 * t, nact);
    }
    ptx::mbar_init(bar_pv_done, 1);
    ptx::mbar_init(bar_o_full, 1);
    ptx::mbar_init(bar_v_fixed, 1);
    ptx::mbar_init(bar_drain, 1);
    misc[1] = 0;
    ptx::fence_mbar_init();
  }
  // Rows R..127 of the Q tile are never loaded: zero them once so the MMA
  // reads defined values (those rows' results are never stored).
  {
    const int zrow_bytes = (kBM - p.R) * 128;
    for (int e = threadIdx.x; e < C::kBoxes * (zrow_bytes >> 4); e += kThreads) {
      const int bx = e / (zrow_bytes >> 4);
      const int off = (e % (zrow_bytes >> 4)) << 4;
      *reinterpret_cast<uint4*>(smem + C::kQOff + bx * kBoxBytes + p.R * 128 + off) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    ptx::fence_proxy_async_smem();
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::tma_prefetch_desc(&tm_q);
    ptx::tma_prefetch_desc(&tm_k);
    ptx::tma_prefetch_desc(&tm_v);
    ptx::tma_prefetch_desc(&tm_o);
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
    int fix_slot = -1;
    uint32_t fix_parity = 0;
    if (lane == 0 && n > 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_first();  // the cache is streamed once
      ptx::mbar_arrive_expect_tx(bar_q_full, C::kBoxes * p.R * 128);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx)
        ptx::tma_load_4d(sQ + bx * kBoxBytes, &tm_q, bar_q_full, bx * 64, hk * p.G, sq0, b, pol_q);
      uint32_t armed = 0, armed_parity = 0;  // per slot: loaded at least once / last parity
      int idx = 0;
      bool ok = true;
      // One ring entry: K (kind 0) or V (kind 1) of KV tile j.
      auto issue = [&](int kind, int j) {
        const int s = idx % C::kStages;
        const uint32_t ph = static_cast<uint32_t>(idx / C::kStages) & 1u;
        ++idx;
        if (aborted() || !ptx::mbar_wait(bar_kv_empty + 8 * s, ph ^ 1u, limit)) {
          fail();
          ok = false;
          return;
        }
        ptx::mbar_arrive_expect_tx(bar_kv_full + 8 * s, C::kTileBytes);
        const CUtensorMap* tm = kind == 0 ? &tm_k : &tm_v;
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          ptx::tma_load_4d(sKV + s * C::kTileBytes + bx * kBoxBytes, tm, bar_kv_full + 8 * s,
                           bx * 64, hk, j * kBN, b, pol_kv);
        armed |= 1u << s;
        armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
        if (kind == 1 && j == jhi - 1) {
          fix_slot = s;
          fix_parity = ph;
        }
      };
      // Ring order = MMA consumption order: K0 K1 | V0 K2 | V1 K3 | ...
      issue(0, jlo);
      if (ok && n > 1) issue(0, jlo + 1);
      for (int r = 0; r < n && ok; ++r) {
        issue(1, jlo + r);
        if (ok && r + 2 < n) issue(0, jlo + r + 2);
      }
      if (!ok) fix_slot = -1;
      // Never leave while a copy of ours may still be writing shared memory.
      ptx::mbar_wait(bar_q_full, 0, drain_limit);
      for (int s = 0; s < C::kStages; ++s)
        if ((armed >> s) & 1u)
          ptx::mbar_wait(bar_kv_full + 8 * s, (armed_parity >> s) & 1u, drain_limit);
    }
    // Zero the V rows past L_b in the last tile (whole warp), then release it.
    fix_slot = __shfl_sync(0xffffffffu, fix_slot, 0);
    fix_parity = __shfl_sync(0xffffffffu, fix_parity, 0);
    if (v_fix && fix_slot >= 0) {
      // The slot's last load is V(jhi - 1): the drain above already waited
      // for it; wait again here so that every lane observes the copy.
      bool w = ptx::mbar_wait(bar_kv_full + 8 * fix_slot, fix_parity, limit);
      w = __all_sync(0xffffffffu, w);
      if (w) {
        const int r0 = L - (jhi - 1) * kBN;                      // first row past L_b
        const int r1 = min(kBN, p.Scache - (jhi - 1) * kBN);     // rows the copy filled
        uint8_t* vt = smem + C::kKVOff + fix_slot * C::kTileBytes;
        const int chunks = (r1 - r0) * 8;                        // 16-byte chunks per box
        for (int e = lane; e < C::kBoxes * chunks; e += 32) {
          const int bx = e / chunks;
          const int off = e % chunks;
          *reinterpret_cast<uint4*>(vt + bx * kBoxBytes + r0 * 128 + off * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_v_fixed);
      } else if (lane == 0) {
        fail();
      }
    }
  } else if (warp == kMmaWarp) {
    // ===================================================== MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, D, false, true);
      bool ok = true;
      // Test hook: wait on the drain barrier, which nothing signals before
      // this thread's own final commit, so the bounded wait must expire.
      if (p.stall_probe && !ptx::mbar_wait(bar_drain, 0, limit)) {
        fail();
        ok = false;
      }
      if (ok && !ptx::mbar_wait(bar_q_full, 0, limit)) {
        fail();
        ok = false;
      }
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
      const uint64_t dq = ptx::smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = ptx::smem_desc_sw128(sKV, 16, 1024);
      const uint64_t dv0 = ptx::smem_desc_sw128(sKV, kBoxBytes, 1024);
      auto issue_s = [&](int buf, int kslot) {
        const uint64_t dk = dk0 + static_cast<uint32_t>((kslot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          ptx::mma_ss(tmem + buf * kBN, dq + off, dk + off, kIdescS, kk > 0 ? 1u : 0u);
        }
        ptx::tc_commit(bar_s_full + 8 * buf);
        ptx::tc_commit(bar_kv_empty + 8 * kslot);
      };
      auto issue_pv = [&](int buf, int vslot, bool accumulate) {
        const uint64_t dv = dv0 + static_cast<uint32_t>((vslot * C::kTileBytes) >> 4);
        const uint32_t acc = accumulate ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          ptx::mma_ts(tmem + kColO, tmem + buf * kBN + kk * 8,
                      dv + static_cast<uint32_t>(kk * 128), kIdescPV, kk > 0 ? 1u : acc);
        ptx::tc_commit(bar_pv_done);
        ptx::tc_commit(bar_kv_empty + 8 * vslot);
      };

      if (ok) {
        int ks = wait_kv();
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
        if (r == n - 1 && v_fix) {
          if (aborted() || !ptx::mbar_wait(bar_v_fixed, 0, limit)) {
            fail();
            break;
          }
          ptx::tc_fence_after();
        }
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
      // Every MMA must have finished before tensor memory is released.
      ptx::tc_commit(bar_drain);
      ptx::mbar_wait(bar_drain, 0, drain_limit);
    }
    __syncwarp();
  } else if (warp < nact) {
    // ===================================================== softmax warps
    const int quad = warp;
    const int row = quad * 32 + lane;
    const int pq = row / p.G;
    const int g = row - pq * p.G;
    const bool valid = row < p.R && pq < nq;
    const int sq = sq0 + pq;
    const int h = hk * p.G + g;
    const int pos = pos0 + pq;
    // Visible keys of this row: [vlo, vhi] (absolute positions).
    const int vlo = p.window > 0 ? max(pos - p.window + 1, 0) : 0;
    const int vhi = p.causal ? min(pos, L - 1)
                             : (p.window > 0 ? min(pos + p.window - 1, L - 1) : L - 1);
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    const float c = p.scale_log2;
    const bool zero_scale = !(c > 0.f);
    const float ce = zero_scale ? 1.f : c;

    float m_use = -INFINITY;  // running max of score * scale * log2(e) (possibly stale)
    float l_run = 0.f;        // running sum of 2^(x - m_use)
    bool ok = true;
    for (int r = 0; r < n; ++r) {
      const int buf = r & 1;
      const uint32_t tS = tmem + lane_base + buf * kBN;
      bool w = ptx::mbar_wait(bar_s_full + 8 * buf, (r >> 1) & 1, limit);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        fail();
        ok = false;
        break;
      }
      ptx::tc_fence_after();

      uint32_t s[kBN];
#pragma unroll
      for (int c0 = 0; c0 < kBN; c0 += 32) ptx::tmem_ld_32x32b_x32(tS + c0, s + c0);
      ptx::tmem_wait_ld();
      ptx::reg_fence<kBN>(s);

      // Rows that are not real (padding) are never stored: skip their mask.
      const int k0 = (jlo + r) * kBN;
      const bool full = !valid || (vlo <= k0 && k0 + kBN - 1 <= vhi);
      if (!full || zero_scale)
        tile::mask_cols(s, valid ? vlo - k0 : 0, valid ? vhi - k0 : kBN - 1, zero_scale);

      const float mx = tile::row_max(s);
      const float m_tile = mx == -INFINITY ? -INFINITY : mx * ce;
      const float m_new = fmaxf(m_use, m_tile);
      float alpha = 1.f;
      bool rescale = false;
      if (r == 0) {
        m_use = m_new;
      } else if (m_new > m_use + kRescaleThreshold) {
        alpha = ptx::ex2_approx(m_use - m_new);  // m_use may be -inf: alpha = 0
        m_use = m_new;
        rescale = true;
      }
      const float neg_base = m_use == -INFINITY ? 0.f : -m_use;
      const float row_sum = tile::exp2_to_bf16(s, ce, neg_base);
      l_run = l_run * alpha + row_sum;
#pragma unroll
      for (int c0 = 0; c0 < kBN / 2; c0 += 32) ptx::tmem_st_32x32b_x32(tS + c0, s + c0);

      // Lazy correction of O: PV(r - 1) must have completed first (S(r) was
      // issued before it, so the S barrier does not imply that).
      if (__any_sync(0xffffffffu, rescale)) {
        bool wp = ptx::mbar_wait(bar_pv_done, (r - 1) & 1, limit);
        wp = __all_sync(0xffffffffu, wp);
        if (!wp) {
          fail();
          ok = false;
          break;
        }
        ptx::tc_fence_after();
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

    // ---- epilogue
    if (ok && n > 0) {
      bool w = ptx::mbar_wait(bar_o_full, 0, limit);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        fail();
        ok = false;
      }
      ptx::tc_fence_after();
    }
    const bool has_o = n > 0;
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    const float lse_row = l_run > 0.f ? ((m_use == -INFINITY ? 0.f : m_use) + __log2f(l_run)) * kLn2
                                      : -INFINITY;
    if (p.splits == 1) {
      // O / l -> bf16 -> shared (swizzled, over the Q tile) -> TMA store.
      if (ok) {
        uint8_t* stage = smem + C::kQOff;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          if (has_o) {
            ptx::tmem_ld_32x32b_x32(tO + c0, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(o);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          tile::stage_bf16_sw128(stage, kBoxBytes, row, c0, o, inv_l);
        }
        ptx::fence_proxy_async_smem();
      }
      ptx::named_bar_sync(1, 32 * nact);
      if (ok && warp == 0 && lane == 0) {
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          ptx::tma_store_4d(&tm_o, sQ + bx * kBoxBytes, bx * 64, hk * p.G, sq0, b);
        ptx::tma_store_commit();
        ptx::tma_store_wait_read();
      }
      if (ok && valid && p.lse != nullptr)
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + sq] = lse_row;
    } else if (ok) {
      // Partial result of this split: O / l (fp32) and its LSE. The
      // tensor-memory loads are warp-collective (.sync.aligned): every lane
      // of the warp issues them; only real rows store.
      const size_t prow = ((static_cast<size_t>(split) * p.B + b) * p.Sq + sq) * p.H + h;
      if (valid)
        p.lse_part[((static_cast<size_t>(split) * p.B + b) * p.H + h) * p.Sq + sq] = lse_row;
      if (has_o) {
        float* dst = p.o_part + prow * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          ptx::tmem_ld_32x32b_x32(tO + c0, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence<32>(o);
          if (valid) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<float4*>(dst + c0 + 4 * u) = make_float4(
                  __uint_as_float(o[4 * u]) * inv_l, __uint_as_float(o[4 * u + 1]) * inv_l,
                  __uint_as_float(o[4 * u + 2]) * inv_l, __uint_as_float(o[4 * u + 3]) * inv_l);
          }
        }
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

// Merges the splits' partial results: one warp per output row (b, s, h).
// Partial rows hold D (padded) floats; out rows hold the real p.D <= D.
// O = sum_i w_i O_i / sum_i w_i and LSE = M + ln(sum_i w_i), with
// w_i = exp(LSE_i - M), M = max_i LSE_i; splits that saw no key (LSE_i = -inf)
// are skipped, and a row no split saw gets O = 0, LSE = -inf.
template <int D>
__global__ void __launch_bounds__(256)
    fa_decode_combine_kernel(const DecodeProblem p, __nv_bfloat16* __restrict__ out) {
  constexpr int kPer = D / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(p.B) * p.Sq * p.H;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (row >= rows) return;
  const int h = static_cast<int>(row % p.H);
  const int sq = static_cast<int>((row / p.H) % p.Sq);
  const int b = static_cast<int>(row / (static_cast<long long>(p.H) * p.Sq));
  auto lse_at = [&](int s) {
    return p.lse_part[((static_cast<size_t>(s) * p.B + b) * p.H + h) * p.Sq + sq];
  };
  float m = -INFINITY;
  for (int s = lane; s < p.splits; s += 32) m = fmaxf(m, lse_at(s));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

  float acc[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) acc[u] = 0.f;
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const float ls = lse_at(s);
      if (ls == -INFINITY) continue;
      const float w = expf(ls - m);
      wsum += w;
      const float* src =
          p.o_part + ((((static_cast<size_t>(s) * p.B + b) * p.Sq + sq) * p.H + h) * D) +
          lane * kPer;
      if constexpr (kPer % 4 == 0) {
#pragma unroll
        for (int u = 0; u < kPer; u += 4) {
          const float4 x = *reinterpret_cast<const float4*>(src + u);
          acc[u] = fmaf(w, x.x, acc[u]);
          acc[u + 1] = fmaf(w, x.y, acc[u + 1]);
          acc[u + 2] = fmaf(w, x.z, acc[u + 2]);
          acc[u + 3] = fmaf(w, x.w, acc[u + 3]);
        }
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = out + static_cast<size_t>(b) * p.so.b + static_cast<size_t>(sq) * p.so.s +
                       static_cast<size_t>(h) * p.so.h + lane * kPer;
  if (lane * kPer + kPer <= p.D) {  // p.D is a multiple of 8: whole groups
    if constexpr (kPer % 4 == 0) {
#pragma unroll
      for (int u = 0; u < kPer; u += 4) {
        uint2 pk;
        pk.x = ptx::pack_bf16x2(acc[u] * inv, acc[u + 1] * inv);
        pk.y = ptx::pack_bf16x2(acc[u + 2] * inv, acc[u + 3] * inv);
        *reinterpret_cast<uint2*>(dst + u) = pk;
      }
    } else {
      *reinterpret_cast<uint32_t*>(dst) = ptx::pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + sq] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

template <int D>
cudaError_t launch_d(const DecodeProblem& p, void* out, const void* q, const void* k,
                     const void* v, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to;
  // The maps carry the real head dim p.D <= D (padding columns: zero-filled
  // on load, clipped on store).
  if (!encode_bshd_tensor_map(&tq, q, p.B, p.Sq, p.H, p.D, p.sq, p.G, p.Pq) ||
      !encode_bshd_tensor_map(&tk, k, p.B, p.Scache, p.Hkv, p.D, p.sk) ||
      !encode_bshd_tensor_map(&tv, v, p.B, p.Scache, p.Hkv, p.D, p.sv) ||
      !encode_bshd_tensor_map(&to, out, p.B, p.Sq, p.H, p.D, p.so, p.G, p.Pq))
    return cudaErrorInvalidValue;
  const long long grid = static_cast<long long>(p.splits) * p.Hkv * p.n_ptiles * p.B;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  static unsigned long long attr_done = 0;
  cudaError_t err = ensure_smem_attr(&attr_done, reinterpret_cast<const void*>(
                                                     &fa_decode_bf16_tc_kernel<D>),
                                     DCfg<D>::kSmemBytes);
  if (err != cudaSuccess) return err;
  fa_decode_bf16_tc_kernel<D><<<static_cast<unsigned>(grid), kThreads, DCfg<D>::kSmemBytes,
                                stream>>>(tq, tk, tv, to, p);
  err = cudaGetLastError();
  if (err != cudaSuccess || p.splits == 1) return err;
  const long long rows = static_cast<long long>(p.B) * p.Sq * p.H;
  const long long cgrid = (rows + 7) / 8;
  if (cgrid > INT_MAX) return cudaErrorInvalidConfiguration;
  DecodeProblem pc = p;  // the combine kernel addresses out with resolved strides
  pc.so = resolve_strides(p.so, p.Sq, p.H, p.D);
  fa_decode_combine_kernel<D><<<static_cast<unsigned>(cgrid), 256, 0, stream>>>(
      pc, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_bf16_tc(const DecodeProblem& p, void* out, const void* q, const void* k,
                                  const void* v, cudaStream_t stream) {
  if (p.D % 8 != 0 || p.D < 8 || p.D > 256) return cudaErrorInvalidValue;
  if (p.D <= 64) return launch_d<64>(p, out, q, k, v, stream);
  if (p.D <= 128) return launch_d<128>(p, out, q, k, v, stream);
  return launch_d<256>(p, out, q, k, v, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
