// fa_fwd_tc.cu -- bf16 fused attention forward on the sm_103a tensor cores.
//
// The operation is `mo.mha.no_cache` (MAX API page "FlashAttentionGPU",
// method `execute`, Steps -1 to 4): O = softmax(mask(scale * Q K^T)) V per
// (batch, query head), Q/K/V/O in BSHD (K/V in BShD for grouped heads). The
// algorithm is the FlashAttention-2 loop of the tiny_flash_attn.py page
// (flash_attn_v2: Q blocks outer, KV blocks inner, running max m and running
// sum l, unnormalised O rescaled by exp(m_old - m_new), one division by l at
// the end), mapped onto Blackwell hardware:
//
//   * one CTA owns two 128-row Q tiles of one (b, h) -- or, for head dims up
//     to 64, one Q tile, with two CTAs per SM -- and streams the K/V tiles
//     they need through a shared-memory ring (TMA, swizzled, straight from
//     BSHD: the Step 0 / Step 4 transposes are the tensor maps' strides);
//   * S = Q K^T and O += P V are tcgen05.mma (bf16 in, fp32 accumulate) with
//     S, P and O resident in tensor memory: S_t at columns [128t, 128t+128),
//     P_t (bf16 pairs) written over the first 64 of them, O_t at
//     [256 + D t, 256 + D (t+1)); one-tile CTAs run a persistent kernel that
//     gives P its own columns and computes S(j+1) during the softmax of j;
//   * warp roles: warps 0-3 and 4-7 are the softmax warpgroups of Q tile 0 and
//     1 (thread = query row = TMEM lane), then one warp issues the MMAs and
//     one the TMA loads. The MMA order S0 S1 | PV0 S0' PV1 S1' | ... lets one
//     tile's softmax overlap the other tile's MMAs; with one Q tile per CTA
//     the two CTAs on an SM overlap the same way, and one CTA's set-up and
//     epilogue overlap the other's KV loop;
//   * softmax in the log2 domain (exp2 of score * scale * log2 e minus the
//     running max), with the rescale of O skipped while the running max grows
//     by less than 2^8 (O and l keep the same stale max, so the final O / l is
//     unchanged);
//   * causal / sliding-window tiles that are entirely hidden are never loaded;
//     only tiles that straddle the mask boundary evaluate the mask per element;
//   * the epilogue writes O / l as bf16 through shared memory and a TMA store
//     (BSHD), and the natural-log LSE per row.
//
// Every mbarrier wait is bounded by the problem's wait limit (global timer):
// on time-out the CTA records kStatusWaitTimeout in the status word, stops
// issuing work, waits (again bounded) for its own copies and MMAs in flight,
// releases its tensor memory and returns.
//
// The debug build (FA_TRACE=1) adds the event trace and bounds guards of
// fa_trace.cuh; in the default build both compile to nothing.
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cmath>

#include "fa_internal.h"
#include "fa_tile.cuh"
#include "fa_trace.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;                          // query rows per Q tile (= TMEM lanes)
constexpr int kBN = tile::kBN;                    // keys per K/V tile
constexpr int kMaxQTiles = 2;                     // Q tiles per CTA: QT = 1 or 2

// Warp roles of a CTA with QT Q tiles: a softmax warpgroup per tile, then
// the MMA warp and the TMA warp.
template <int QT>
struct Roles {
  static constexpr int kSoftmaxWarps = 4 * QT;
  static constexpr int kMmaWarp = kSoftmaxWarps;
  static constexpr int kLoadWarp = kSoftmaxWarps + 1;
  static constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
  // One CTA of two tiles fills an SM's tensor memory; two CTAs of one tile
  // share it (256 columns each: S 128, O up to 128).
  static constexpr uint32_t kTmemCols = QT == 2 ? 512 : 256;
  static constexpr int kCtasPerSm = 3 - QT;
};
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr unsigned long long kDrainExtraNs = 100000000ull;  // 100 ms

// Tiles of 128 rows x D bf16 columns are held as TMA boxes of [128][64] with
// the 128-byte swizzle (D = 64, 128) or, for D = 96, of [128][32] with the
// 64-byte swizzle (three boxes: the MMAs then run with K = 96 and N = 96, no
// padding columns).
template <int D, int QT>
struct Cfg {
  static_assert(D == 64 || D == 96 || D == 128, "head dim");
  static_assert(QT == 2 || D <= 64, "one Q tile per CTA is built for D <= 64");
  static constexpr int kBoxCols = D == 96 ? 32 : 64;
  static constexpr int kRowBytes = kBoxCols * 2;          // bytes of one box row (= swizzle span)
  static constexpr int kBoxBytes = kBM * kRowBytes;
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kKPerBox = kBoxCols / 16;          // MMA K steps of 16 per box
  static constexpr uint32_t kSwizzle = D == 96 ? ptx::kSwizzle64B : ptx::kSwizzle128B;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;  // one [128][D] bf16 tile
  // K/V ring slots (one Q tile: small enough for two CTAs per SM)
  static constexpr int kStages = QT == 1 ? 5 : (D == 128 ? 4 : 6);
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + QT * kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // q_full[2] kv_full[S] kv_empty[S] s_full[2] p_full[2] o_full[2] drain
  static constexpr int kNumBars = 2 + 2 * kStages + 2 + 2 + 2 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack for 1 KB alignment
  static constexpr uint32_t kColO = 128 * QT;              // O_t at kColO + t * D
  static_assert(kColO + QT * D <= Roles<QT>::kTmemCols, "tensor memory");
  static_assert(Roles<QT>::kCtasPerSm * (kSmemBytes + 1024) <= 228 * 1024, "shared memory");
};

// Visibility bounds of query row i (keys lo..hi inclusive may be visible).
struct RowBounds {
  int lo, hi;
};

__device__ __forceinline__ RowBounds row_bounds(const FwdProblem& p, int i) {
  RowBounds r;
  r.lo = p.window > 0 ? i - p.window + 1 : INT_MIN;
  r.hi = p.causal ? min(i, p.S - 1) : (p.window > 0 ? min(i + p.window - 1, p.S - 1) : p.S - 1);
  return r;
}

template <int D, int QT>
__global__ void __launch_bounds__(Roles<QT>::kThreads, Roles<QT>::kCtasPerSm)
    fa_fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_o, const FwdProblem p,
                          int num_qblocks) {
  using C = Cfg<D, QT>;
  constexpr int kSoftmaxWarps = Roles<QT>::kSoftmaxWarps;
  constexpr int kMmaWarp = Roles<QT>::kMmaWarp;
  constexpr int kLoadWarp = Roles<QT>::kLoadWarp;
  constexpr uint32_t kTmemCols = Roles<QT>::kTmemCols;
  (void)kSoftmaxWarps;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kQOff;
  const uint32_t sKV = base + C::kKVOff;
  const uint32_t bars = base + C::kBarOff;
  const uint32_t bar_q_full = bars;                              // + 8 t
  const uint32_t bar_kv_full = bars + 8 * 2;                     // + 8 s
  const uint32_t bar_kv_empty = bars + 8 * (2 + C::kStages);     // + 8 s
  const uint32_t bar_s_full = bars + 8 * (2 + 2 * C::kStages);   // + 8 t
  const uint32_t bar_p_full = bar_s_full + 16;                   // + 8 t
  const uint32_t bar_o_full = bar_p_full + 16;                   // + 8 t
  const uint32_t bar_drain = bar_o_full + 16;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
  // misc[0]: tensor-memory base address, misc[1]: abort flag

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  namespace tr = trace;
  const int trace_role = warp == kLoadWarp ? tr::kRoleProducer
                         : warp == kMmaWarp ? tr::kRoleMma
                                            : tr::softmax_role(warp);
  tr::Recorder rec(p.trace, p.trace_ctas, trace_role, lane == 0);
  if (warp == kLoadWarp) rec(tr::kCtaStart, tr::sm_id());

  // ---- work item: heaviest (last) query blocks first
  const int per_qb = p.H * p.B;
  const int qb = num_qblocks - 1 - static_cast<int>(blockIdx.x / per_qb);
  const int rem = static_cast<int>(blockIdx.x % per_qb);
  const int h = rem % p.H;
  const int b = rem / p.H;
  const int hk = h / (p.H / p.Hkv);

  // KV tile range [lo_t, hi_t) of each Q tile; empty when the tile is past S
  // (and for tile 1 of a one-tile CTA).
  int q0[kMaxQTiles], lo[kMaxQTiles], hi[kMaxQTiles];
#pragma unroll
  for (int t = 0; t < kMaxQTiles; ++t) {
    q0[t] = qb * (QT * kBM) + t * kBM;
    if (t < QT && q0[t] < p.S) {
      // Window without the causal mask: keys up to the last row + W - 1.
      const int kv_end = p.causal ? min(p.S, q0[t] + kBM)
                                  : (p.window > 0 ? min(p.S, q0[t] + kBM - 1 + p.window) : p.S);
      const int kv_begin = p.window > 0 ? max(0, q0[t] - p.window + 1) : 0;
      lo[t] = kv_begin / kBN;
      hi[t] = (kv_end + kBN - 1) / kBN;
    } else {
      lo[t] = hi[t] = 0;
    }
  }
  const int jlo = lo[0];
  const int jhi = max(hi[0], hi[1]);
  const unsigned long long limit = p.wait_limit_ns;
  const unsigned long long drain_limit = limit + kDrainExtraNs;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int t = 0; t < kMaxQTiles; ++t) {
      ptx::mbar_init(bar_q_full + 8 * t, 1);
      ptx::mbar_init(bar_s_full + 8 * t, 1);
      ptx::mbar_init(bar_p_full + 8 * t, 4);  // one arrival per softmax warp
      ptx::mbar_init(bar_o_full + 8 * t, 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar_kv_full + 8 * s, 1);
      ptx::mbar_init(bar_kv_empty + 8 * s, 1);
    }
    ptx::mbar_init(bar_drain, 1);
    misc[1] = 0;
    ptx::fence_mbar_init();
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
    if (lane == 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
#pragma unroll
      for (int t = 0; t < QT; ++t) {
        if (lo[t] < hi[t]) {
          ptx::mbar_arrive_expect_tx(bar_q_full + 8 * t, C::kTileBytes);
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            ptx::tma_load_4d(sQ + t * C::kTileBytes + bx * C::kBoxBytes, &tm_q, bar_q_full + 8 * t,
                             bx * C::kBoxCols, h, q0[t], b, pol_q);
          rec(tr::kQLoadIssued, t);
        }
      }
      uint32_t armed = 0, armed_parity = 0;  // per slot: bit set once loaded / last parity
      int idx = 0;
      bool ok = true;
      // Ring order: K_jlo, V_jlo, K_jlo+1, V_jlo+1, ...
      for (int j = jlo; j < jhi && ok; ++j) {
        for (int kind = 0; kind < 2; ++kind, ++idx) {
          const int s = idx % C::kStages;
          const uint32_t ph = static_cast<uint32_t>(idx / C::kStages) & 1u;
          if (aborted() || !ptx::mbar_wait(bar_kv_empty + 8 * s, ph ^ 1u, limit)) {
            fail();
            ok = false;
            break;
          }
          // A tile starting past the last key would be a planning error.
          tr::guard(j * kBN < p.S, p.status, kStatusBoundsGuard);
          ptx::mbar_arrive_expect_tx(bar_kv_full + 8 * s, C::kTileBytes);
          const CUtensorMap* tm = kind == 0 ? &tm_k : &tm_v;
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            ptx::tma_load_4d(sKV + s * C::kTileBytes + bx * C::kBoxBytes, tm, bar_kv_full + 8 * s,
                             bx * C::kBoxCols, hk, j * kBN, b, pol_kv);
          rec(kind == 0 ? tr::kKLoadIssued : tr::kVLoadIssued, j);
          armed |= 1u << s;
          armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
        }
      }
      // Never leave while a copy of ours may still be writing shared memory.
#pragma unroll
      for (int t = 0; t < QT; ++t)
        if (lo[t] < hi[t]) ptx::mbar_wait(bar_q_full + 8 * t, 0, drain_limit);
      for (int s = 0; s < C::kStages; ++s)
        if ((armed >> s) & 1u) ptx::mbar_wait(bar_kv_full + 8 * s, (armed_parity >> s) & 1u, drain_limit);
    }
  } else if (warp == kMmaWarp) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, D, false, true);
      bool ok = true;
      // Test hook: wait on the drain barrier, which nothing signals before
      // this thread's own final commit, so the bounded wait must expire.
      if (p.stall_probe && !ptx::mbar_wait(bar_drain, 0, limit)) {
        fail();
        ok = false;
      }
#pragma unroll
      for (int t = 0; t < QT; ++t)
        if (ok && lo[t] < hi[t] && !ptx::mbar_wait(bar_q_full + 8 * t, 0, limit)) {
          fail();
          ok = false;
        }
      rec(tr::kQReady, 0);
      auto in_tile = [&](int t, int j) { return j >= lo[t] && j < hi[t]; };
      // Wait for ring entry idx; returns its slot or -1 on time-out.
      auto wait_kv = [&](int idx) -> int {
        const int s = idx % C::kStages;
        const uint32_t ph = static_cast<uint32_t>(idx / C::kStages) & 1u;
        if (aborted() || !ptx::mbar_wait(bar_kv_full + 8 * s, ph, limit)) {
          fail();
          return -1;
        }
        ptx::tc_fence_after();
        return s;
      };
      // K-major Q and K: 8-row groups 8 box rows apart. MN-major V: atoms
      // of kBoxCols columns one box apart.
      const uint64_t dq0 = ptx::smem_desc(sQ, 16, 8 * C::kRowBytes, C::kSwizzle);
      const uint64_t dk0 = ptx::smem_desc(sKV, 16, 8 * C::kRowBytes, C::kSwizzle);
      const uint64_t dv0 = ptx::smem_desc(sKV, C::kBoxBytes, 8 * C::kRowBytes, C::kSwizzle);
      auto issue_s = [&](int t, int kslot, int j) {
        const uint64_t dq = dq0 + static_cast<uint32_t>((t * C::kTileBytes) >> 4);
        const uint64_t dk = dk0 + static_cast<uint32_t>((kslot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>(
              ((kk / C::kKPerBox) * C::kBoxBytes + (kk % C::kKPerBox) * 32) >> 4);
          ptx::mma_ss(tmem + t * kBN, dq + off, dk + off, kIdescS, kk > 0 ? 1u : 0u);
        }
        ptx::tc_commit(bar_s_full + 8 * t);
        rec(tr::kSIssued, (t << 16) | j);
      };
      auto issue_pv = [&](int t, int vslot, bool accumulate, int j) {
        const uint64_t dv = dv0 + static_cast<uint32_t>((vslot * C::kTileBytes) >> 4);
        const uint32_t acc = accumulate ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          ptx::mma_ts(tmem + C::kColO + t * D, tmem + t * kBN + kk * 8,
                      dv + static_cast<uint32_t>(kk * (16 * C::kRowBytes >> 4)), kIdescPV,
                      kk > 0 ? 1u : acc);
        rec(tr::kPvIssued, (t << 16) | j);
      };
      uint32_t p_phase[kMaxQTiles] = {0u, 0u};
      auto wait_p = [&](int t, int j) -> bool {
        if (aborted() || !ptx::mbar_wait(bar_p_full + 8 * t, p_phase[t], limit)) {
          fail();
          return false;
        }
        p_phase[t] ^= 1u;
        ptx::tc_fence_after();
        rec(tr::kPSeen, (t << 16) | j);
        return true;
      };

      if (ok) {
        const int ks = wait_kv(0);
        if (ks < 0) {
          ok = false;
        } else {
#pragma unroll
          for (int t = 0; t < QT; ++t)
            if (in_tile(t, jlo)) issue_s(t, ks, jlo);
          ptx::tc_commit(bar_kv_empty + 8 * ks);
        }
      }
      for (int j = jlo; ok && j < jhi; ++j) {
        const int rel = j - jlo;
        const int vs = wait_kv(2 * rel + 1);
        if (vs < 0) break;
        if (in_tile(0, j)) {
          if (!wait_p(0, j)) break;
          issue_pv(0, vs, j > lo[0], j);
          if (j == hi[0] - 1) ptx::tc_commit(bar_o_full);
        }
        const bool has_next = j + 1 < jhi;
        int ks = -1;
        if (has_next) {
          ks = wait_kv(2 * rel + 2);
          if (ks < 0) break;
          if (in_tile(0, j + 1)) issue_s(0, ks, j + 1);
        }
        if (QT > 1 && in_tile(1, j)) {
          if (!wait_p(1, j)) break;
          issue_pv(1, vs, j > lo[1], j);
          if (j == hi[1] - 1) ptx::tc_commit(bar_o_full + 8);
        }
        ptx::tc_commit(bar_kv_empty + 8 * vs);
        if (has_next) {
          if (QT > 1 && in_tile(1, j + 1)) issue_s(1, ks, j + 1);
          ptx::tc_commit(bar_kv_empty + 8 * ks);
        }
      }
      // Every MMA must have finished before tensor memory is released.
      ptx::tc_commit(bar_drain);
      ptx::mbar_wait(bar_drain, 0, drain_limit);
      rec(tr::kMmaDrained, 0);
    }
    __syncwarp();
  } else {
    // ===================================================== softmax warpgroups
    const int t = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    // This warpgroup's tile, selected without run-time array indexing.
    const int tq0 = t == 0 ? q0[0] : q0[1];
    const int tlo = t == 0 ? lo[0] : lo[1];
    const int thi = t == 0 ? hi[0] : hi[1];
    const int i = tq0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * kBN;
    const uint32_t tO = tmem + lane_base + C::kColO + t * D;
    const float c = p.scale_log2;
    const RowBounds rb = row_bounds(p, i);
    // A zero scale makes every visible score 0: use 0 as the score and 1 as
    // the multiplier.
    const bool zero_scale = !(c > 0.f);
    const float ce = zero_scale ? 1.f : c;

    float m_use = -INFINITY;  // running max of score * scale * log2(e) (possibly stale)
    float l_run = 0.f;        // running sum of 2^(x - m_use)
    bool ok = true;
    uint32_t s_phase = 0;
    for (int j = tlo; j < thi; ++j) {
      bool w = ptx::mbar_wait(bar_s_full + 8 * t, s_phase, limit);
      s_phase ^= 1u;
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        fail();
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      rec(tr::kSReady, j);

      uint32_t r[kBN];
      float pm[kBN / 32];  // maximum of each 32 columns, reduced by the load
#pragma unroll
      for (int c0 = 0; c0 < kBN; c0 += 32) ptx::tmem_ld_max_32x32b_x32(tS + c0, r + c0, &pm[c0 / 32]);
      ptx::tmem_wait_ld();
      ptx::reg_fence<kBN>(r);
      tile::float_fence<kBN / 32>(pm);
      rec(tr::kSLoaded, j);

      const int k0 = j * kBN;
      bool full = k0 + kBN <= p.S;
      if (p.causal) full = full && (k0 + kBN - 1 <= tq0);
      if (p.window > 0) full = full && (tq0 + kBM - 1 - k0 < p.window);
      if (p.window > 0 && !p.causal) full = full && (k0 + kBN - 1 - tq0 < p.window);
      const int vlo = rb.lo == INT_MIN ? INT_MIN : rb.lo - k0;
      const int vhi = rb.hi - k0;

      // Tiles that straddle the mask boundary (or a zero scale): hide the
      // invisible scores in place, then every tile takes the same path.
      if (!full || zero_scale) tile::mask_cols(r, vlo, vhi, zero_scale);

      // Row maximum of the (visible) scores: from the loads' reductions when
      // every score is visible, else over the masked registers.
      float mx;
      if (full && !zero_scale)
        mx = tile::max_of(pm);
      else
        mx = tile::row_max(r);
      if (FA_TRACE) {
        asm volatile("" ::"f"(mx));
        rec(tr::kMaxDone, j);
      }
      const float m_tile = mx == -INFINITY ? -INFINITY : mx * ce;
      const float m_new = fmaxf(m_use, m_tile);
      const bool first = j == tlo;
      float alpha = 1.f;
      bool rescale = false;
      if (first) {
        m_use = m_new;
      } else if (m_new > m_use + kRescaleThreshold) {
        alpha = ptx::ex2_approx(m_use - m_new);  // m_use may be -inf: alpha = 0
        m_use = m_new;
        rescale = true;
      }
      const float neg_base = m_use == -INFINITY ? 0.f : -m_use;

      // P = 2^(x - m_use) (hidden scores are -inf and give 0) as bf16 pairs
      // written over S, and the row sum.
      const float row_sum = tile::exp2_to_bf16(r, ce, neg_base);
      l_run = l_run * alpha + row_sum;
      if (FA_TRACE) {
        asm volatile("" ::"f"(l_run), "r"(r[0]), "r"(r[63]));
        rec(tr::kExpDone, j);
      }
#pragma unroll
      for (int c0 = 0; c0 < kBN / 2; c0 += 32) ptx::tmem_st_32x32b_x32(tS + c0, r + c0);

      // Lazy correction of the O accumulator (previous PV has completed:
      // the S MMA this iteration waited for was issued after it).
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
      if (lane == 0) ptx::mbar_arrive(bar_p_full + 8 * t);
      rec(tr::kPReady, j | (rescale ? 1u << 23 : 0u));
    }

    // ---- epilogue: O / l -> bf16 -> shared (swizzled) -> TMA store; LSE.
    const bool has_work = tlo < thi;
    if (ok && has_work) {
      bool w = ptx::mbar_wait(bar_o_full + 8 * t, 0, limit);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        fail();
        ok = false;
      }
    }
    // A store of rows that start past S would be a planning error.
    const bool do_store = ok && has_work && tr::guard(tq0 < p.S, p.status, kStatusBoundsGuard);
    if (do_store) {
      rec(tr::kEpilogueStart, 0);
      ptx::tc_fence_after();
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      uint8_t* stage = smem + C::kQOff + t * C::kTileBytes;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        ptx::tmem_ld_32x32b_x32(tO + c0, o);
        ptx::tmem_wait_ld();
        ptx::reg_fence<32>(o);
        if (D == 96)
          tile::stage_bf16_sw64(stage, C::kBoxBytes, row, c0, o, inv_l);
        else
          tile::stage_bf16_sw128(stage, C::kBoxBytes, row, c0, o, inv_l);
      }
      ptx::fence_proxy_async_smem();
    }
    ptx::named_bar_sync(1 + t, 128);
    if (do_store && quad == 0 && lane == 0) {
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx)
        ptx::tma_store_4d(&tm_o, sQ + t * C::kTileBytes + bx * C::kBoxBytes, bx * C::kBoxCols, h,
                          tq0, b);
      ptx::tma_store_commit();
      ptx::tma_store_wait_read();
    }
    if (do_store && p.lse != nullptr && i < p.S) {
      const float m_fin = m_use == -INFINITY ? 0.f : m_use;
      const long long idx = (static_cast<long long>(b) * p.H + h) * p.S + i;
      const long long lse_limit =
          p.lse_limit > 0 ? p.lse_limit : static_cast<long long>(p.B) * p.H * p.S;
      if (tr::guard(idx < lse_limit, p.status, kStatusBoundsGuard))
        p.lse[idx] = (m_fin + __log2f(l_run)) * kLn2;
    }
    if (do_store) rec(tr::kEpilogueEnd, 0);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- persistent
// One Q tile per CTA (head dims up to 64), persistent CTAs, one per resident
// slot, each walking a sequence of items (query blocks). With one tile of at
// most 64 columns, 64 of the CTA's 256 tensor-memory columns are left over
// after S (128) and O (64): P gets them to itself, so S(j+1) no longer waits
// for PV(j) to have read P(j) out of S's columns. The MMA thread issues
// S(j+1) as soon as the softmax has loaded S(j) into registers, and the
// tensor core computes it while the softmax of step j runs; the softmax then
// waits for PV(j-1) only before it overwrites P (and before a rescale of O).
// Q is double-buffered, so the next item's Q is loaded during the current
// item, and the first S of an item is computed during the previous item's
// epilogue; the epilogue hands O back to the MMA thread (o_free) as soon as
// it has read it out of tensor memory. The ring, the phases and the counts
// carry on from one item to the next. Used for every launch with a head dim
// up to 64, at every length; with fewer items than resident slots each CTA
// takes one item and still gains the early S.
//
// TMEM columns: S [0, 128), O [128, 128 + D), P [128 + D, 128 + D + 64).
template <int D>
struct PCfg {
  static_assert(D == 64, "the persistent one-tile kernel is built for the 64-column layout");
  using Geo = Cfg<D, 1>;  // TMA box geometry of the 64-column tiles
  static constexpr int kBoxCols = Geo::kBoxCols;
  static constexpr int kRowBytes = Geo::kRowBytes;
  static constexpr int kBoxBytes = Geo::kBoxBytes;
  static constexpr int kBoxes = Geo::kBoxes;
  static constexpr int kKPerBox = Geo::kKPerBox;
  static constexpr uint32_t kSwizzle = Geo::kSwizzle;
  static constexpr int kTileBytes = Geo::kTileBytes;
  static constexpr int kQBufs = 2;
  static constexpr int kStages = 4;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQBufs * kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // q_full[2] q_free[2] kv_full[S] kv_empty[S] s_full s_free p_full pv_done
  // o_full o_free drain
  static constexpr int kNumBars = 2 * kQBufs + 2 * kStages + 7;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack for 1 KB alignment
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = kBN;
  static constexpr uint32_t kColP = kBN + D;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr int kThreads = 6 * 32;  // 4 softmax warps, MMA warp, TMA warp
  static constexpr int kMmaWarp = 4;
  static constexpr int kLoadWarp = 5;
  static constexpr int kCtasPerSm = 2;
  static_assert(kColP + kBN / 2 <= kTmemCols, "tensor memory");
  static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 228 * 1024, "shared memory");
};

// One work item: the Q tile of query block qb of head h, batch b (the
// heaviest -- last -- query blocks first), and its KV tile range [lo, hi).
struct QItem {
  int b, h, hk, q0, lo, hi;
};

__device__ __forceinline__ QItem decode_qitem(const FwdProblem& p, int item, int num_qblocks) {
  QItem w;
  const int per_qb = p.H * p.B;
  const int qb = num_qblocks - 1 - item / per_qb;
  const int rem = item % per_qb;
  w.h = rem % p.H;
  w.b = rem / p.H;
  w.hk = w.h / (p.H / p.Hkv);
  w.q0 = qb * kBM;
  if (w.q0 < p.S) {
    // Window without the causal mask: keys up to the last row + W - 1.
    const int kv_end = p.causal ? min(p.S, w.q0 + kBM)
                                : (p.window > 0 ? min(p.S, w.q0 + kBM - 1 + p.window) : p.S);
    const int kv_begin = p.window > 0 ? max(0, w.q0 - p.window + 1) : 0;
    w.lo = kv_begin / kBN;
    w.hi = (kv_end + kBN - 1) / kBN;
  } else {
    w.lo = w.hi = 0;
  }
  return w;
}

// Persistent schedule: item number of this CTA's k-th item, or -1. The CTAs
// take the items in rounds, snake order: round r gives CTA g item r * C + g
// for even r and r * C + C - 1 - g for odd r, so the heavy items of one round
// and the light ones of the next pair up.
__device__ __forceinline__ int qitem_at(int k, int n_items) {
  const int C = static_cast<int>(gridDim.x);
  const int pos = (k & 1) ? C - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  const long long it = static_cast<long long>(k) * C + pos;
  return it < n_items ? static_cast<int>(it) : -1;
}

// Walks this CTA's KV steps in order, across its items (items with no KV
// tile are skipped). u counts the items with work (their Q buffer is u & 1).
struct StepCursor {
  int k = -1, u = -1, j = 0;
  QItem w;
  bool valid = false;
  __device__ __forceinline__ void next_item(const FwdProblem& p, int n_items, int nqb) {
    for (;;) {
      const int item = qitem_at(++k, n_items);
      if (item < 0) {
        valid = false;
        return;
      }
      w = decode_qitem(p, item, nqb);
      if (w.lo < w.hi) break;
    }
    ++u;
    j = w.lo;
    valid = true;
  }
  __device__ __forceinline__ void advance(const FwdProblem& p, int n_items, int nqb) {
    if (++j >= w.hi) next_item(p, n_items, nqb);
  }
  __device__ __forceinline__ bool first() const { return j == w.lo; }
  __device__ __forceinline__ bool last() const { return j == w.hi - 1; }
};

template <int D>
__global__ void __launch_bounds__(PCfg<D>::kThreads, PCfg<D>::kCtasPerSm)
    fa_fwd_bf16_tc_persistent_kernel(const __grid_constant__ CUtensorMap tm_q,
                                     const __grid_constant__ CUtensorMap tm_k,
                                     const __grid_constant__ CUtensorMap tm_v,
                                     const __grid_constant__ CUtensorMap tm_o, const FwdProblem p,
                                     int num_qblocks) {
  using C = PCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kQOff;
  const uint32_t sKV = base + C::kKVOff;
  const uint32_t bars = base + C::kBarOff;
  const uint32_t bar_q_full = bars;                             // + 8 buffer
  const uint32_t bar_q_free = bars + 8 * C::kQBufs;             // + 8 buffer
  const uint32_t bar_kv_full = bars + 16 * C::kQBufs;           // + 8 s
  const uint32_t bar_kv_empty = bar_kv_full + 8 * C::kStages;   // + 8 s
  const uint32_t bar_s_full = bar_kv_empty + 8 * C::kStages;    // S(n) in tensor memory
  const uint32_t bar_s_free = bar_s_full + 8;                   // S(n) read by the softmax
  const uint32_t bar_p_full = bar_s_free + 8;                   // P(n) stored, O corrected
  const uint32_t bar_pv_done = bar_p_full + 8;                  // PV(n) completed
  const uint32_t bar_o_full = bar_pv_done + 8;                  // item's last PV completed
  const uint32_t bar_o_free = bar_o_full + 8;                   // item's O read out
  const uint32_t bar_drain = bar_o_free + 8;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
  // misc[0]: tensor-memory base address, misc[1]: abort flag, misc[2]: a
  // softmax warp timed out (read by all four at an item's epilogue barrier)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  namespace tr = trace;
  const int trace_role = warp == C::kLoadWarp ? tr::kRoleProducer
                         : warp == C::kMmaWarp ? tr::kRoleMma
                                               : tr::softmax_role(warp);
  tr::Recorder rec(p.trace, p.trace_ctas, trace_role, lane == 0);
  if (warp == C::kLoadWarp) rec(tr::kCtaStart, tr::sm_id());

  const int n_items = num_qblocks * p.H * p.B;
  const unsigned long long limit = p.wait_limit_ns;
  const unsigned long long drain_limit = limit + kDrainExtraNs;

  if (threadIdx.x == 0) {
    for (int b = 0; b < C::kQBufs; ++b) {
      ptx::mbar_init(bar_q_full + 8 * b, 1);
      ptx::mbar_init(bar_q_free + 8 * b, 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar_kv_full + 8 * s, 1);
      ptx::mbar_init(bar_kv_empty + 8 * s, 1);
    }
    ptx::mbar_init(bar_s_full, 1);
    ptx::mbar_init(bar_s_free, 4);  // one arrival per softmax warp
    ptx::mbar_init(bar_p_full, 4);
    ptx::mbar_init(bar_pv_done, 1);
    ptx::mbar_init(bar_o_full, 1);
    ptx::mbar_init(bar_o_free, 4);
    ptx::mbar_init(bar_drain, 1);
    misc[1] = 0;
    misc[2] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    ptx::tma_prefetch_desc(&tm_q);
    ptx::tma_prefetch_desc(&tm_k);
    ptx::tma_prefetch_desc(&tm_v);
    ptx::tma_prefetch_desc(&tm_o);
  }
  if (warp == C::kMmaWarp) {
    ptx::tmem_alloc(base + C::kMiscOff, C::kTmemCols);
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

  if (warp == C::kLoadWarp) {
    // ===================================================== TMA producer
    if (lane == 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
      uint32_t armed = 0, armed_parity = 0;  // per slot: bit set once loaded / last parity
      int idx = 0;                           // ring entries so far: K(n) at 2n, V(n) at 2n + 1
      int nq = 0;                            // Q loads so far (item u into buffer u & 1)
      bool ok = true;
      for (int k = 0, item; ok && (item = qitem_at(k, n_items)) >= 0; ++k) {
        const QItem w = decode_qitem(p, item, num_qblocks);
        if (w.lo >= w.hi) continue;
        // Buffer qb last held item nq - 2, whose O was staged over it.
        const int qb = nq & 1;
        if (nq >= C::kQBufs &&
            (aborted() || !ptx::mbar_wait(bar_q_free + 8 * qb,
                                          static_cast<uint32_t>((nq >> 1) - 1) & 1u, limit))) {
          fail();
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(bar_q_full + 8 * qb, C::kTileBytes);
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          ptx::tma_load_4d(sQ + qb * C::kTileBytes + bx * C::kBoxBytes, &tm_q, bar_q_full + 8 * qb,
                           bx * C::kBoxCols, w.h, w.q0, w.b, pol_q);
        ++nq;
        rec(tr::kQLoadIssued, qb);
        for (int j = w.lo; j < w.hi && ok; ++j) {
          for (int kind = 0; kind < 2; ++kind, ++idx) {
            const int s = idx % C::kStages;
            const uint32_t ph = static_cast<uint32_t>(idx / C::kStages) & 1u;
            if (aborted() || !ptx::mbar_wait(bar_kv_empty + 8 * s, ph ^ 1u, limit)) {
              fail();
              ok = false;
              break;
            }
            // A tile starting past the last key would be a planning error.
            tr::guard(j * kBN < p.S, p.status, kStatusBoundsGuard);
            ptx::mbar_arrive_expect_tx(bar_kv_full + 8 * s, C::kTileBytes);
            const CUtensorMap* tm = kind == 0 ? &tm_k : &tm_v;
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
              ptx::tma_load_4d(sKV + s * C::kTileBytes + bx * C::kBoxBytes, tm,
                               bar_kv_full + 8 * s, bx * C::kBoxCols, w.hk, j * kBN, w.b, pol_kv);
            rec(kind == 0 ? tr::kKLoadIssued : tr::kVLoadIssued, j);
            armed |= 1u << s;
            armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
          }
        }
      }
      // Never leave while a copy of ours may still be writing shared memory.
      for (int qb = 0; qb < C::kQBufs; ++qb) {
        const int uses = (nq + C::kQBufs - 1 - qb) / C::kQBufs;
        if (uses > 0)
          ptx::mbar_wait(bar_q_full + 8 * qb, static_cast<uint32_t>(uses - 1) & 1u, drain_limit);
      }
      for (int s = 0; s < C::kStages; ++s)
        if ((armed >> s) & 1u) ptx::mbar_wait(bar_kv_full + 8 * s, (armed_parity >> s) & 1u, drain_limit);
    }
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, D, false, true);
      bool ok = true;
      // Test hook: wait on the drain barrier, which nothing signals before
      // this thread's own final commit, so the bounded wait must expire.
      if (p.stall_probe && !ptx::mbar_wait(bar_drain, 0, limit)) {
        fail();
        ok = false;
      }
      auto wait_bar = [&](uint32_t bar, uint32_t parity) -> bool {
        if (aborted() || !ptx::mbar_wait(bar, parity, limit)) {
          fail();
          return false;
        }
        ptx::tc_fence_after();
        return true;
      };
      // Wait for ring entry idx; returns its slot or -1 on time-out.
      auto wait_kv = [&](int idx) -> int {
        const int s = idx % C::kStages;
        return wait_bar(bar_kv_full + 8 * s, static_cast<uint32_t>(idx / C::kStages) & 1u) ? s : -1;
      };
      // K-major Q and K: 8-row groups 8 box rows apart. MN-major V: atoms
      // of kBoxCols columns one box apart.
      const uint64_t dq0 = ptx::smem_desc(sQ, 16, 8 * C::kRowBytes, C::kSwizzle);
      const uint64_t dk0 = ptx::smem_desc(sKV, 16, 8 * C::kRowBytes, C::kSwizzle);
      const uint64_t dv0 = ptx::smem_desc(sKV, C::kBoxBytes, 8 * C::kRowBytes, C::kSwizzle);

      // cs walks the steps whose S is issued, one ahead of cp, whose PV is.
      StepCursor cs, cp;
      cs.next_item(p, n_items, num_qblocks);
      cp = cs;
      int ns = 0;  // S MMAs issued (global step count)
      // S(ns) = Q K(j)^T into S's columns; an item's first S waits for its Q.
      auto issue_s = [&]() -> bool {
        const int qb = cs.u & 1;
        if (cs.first()) {
          if (!wait_bar(bar_q_full + 8 * qb, static_cast<uint32_t>(cs.u >> 1) & 1u)) return false;
          rec(tr::kQReady, 0);
        }
        const int ks = wait_kv(2 * ns);
        if (ks < 0) return false;
        const uint64_t dq = dq0 + static_cast<uint32_t>((qb * C::kTileBytes) >> 4);
        const uint64_t dk = dk0 + static_cast<uint32_t>((ks * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>(
              ((kk / C::kKPerBox) * C::kBoxBytes + (kk % C::kKPerBox) * 32) >> 4);
          ptx::mma_ss(tmem + C::kColS, dq + off, dk + off, kIdescS, kk > 0 ? 1u : 0u);
        }
        ptx::tc_commit(bar_s_full);
        ptx::tc_commit(bar_kv_empty + 8 * ks);
        rec(tr::kSIssued, cs.j);
        ++ns;
        cs.advance(p, n_items, num_qblocks);
        return true;
      };
      if (ok && cs.valid) ok = issue_s();
      for (int n = 0; ok && cp.valid; ++n) {
        // The next S, over S(n), as soon as the softmax has read S(n).
        if (cs.valid && !(wait_bar(bar_s_free, static_cast<uint32_t>(n) & 1u) && issue_s())) {
          ok = false;
          break;
        }
        // PV(n) once P(n) is stored; an item's first PV (which starts O
        // afresh) also waits until the previous item's O has been read out.
        if (!wait_bar(bar_p_full, static_cast<uint32_t>(n) & 1u)) {
          ok = false;
          break;
        }
        rec(tr::kPSeen, cp.j);
        const int vs = wait_kv(2 * n + 1);
        if (vs < 0 || (cp.first() && cp.u > 0 &&
                       !wait_bar(bar_o_free, static_cast<uint32_t>(cp.u - 1) & 1u))) {
          ok = false;
          break;
        }
        const uint64_t dv = dv0 + static_cast<uint32_t>((vs * C::kTileBytes) >> 4);
        const uint32_t acc = cp.first() ? 0u : 1u;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          ptx::mma_ts(tmem + C::kColO, tmem + C::kColP + kk * 8,
                      dv + static_cast<uint32_t>(kk * (16 * C::kRowBytes >> 4)), kIdescPV,
                      kk > 0 ? 1u : acc);
        ptx::tc_commit(bar_pv_done);
        ptx::tc_commit(bar_kv_empty + 8 * vs);
        if (cp.last()) ptx::tc_commit(bar_o_full);
        rec(tr::kPvIssued, cp.j);
        cp.advance(p, n_items, num_qblocks);
      }
      // Every MMA must have finished before tensor memory is released.
      ptx::tc_commit(bar_drain);
      ptx::mbar_wait(bar_drain, 0, drain_limit);
      rec(tr::kMmaDrained, 0);
    }
    __syncwarp();
  } else {
    // ===================================================== softmax warpgroup
    const int row = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kColS;
    const uint32_t tO = tmem + lane_base + C::kColO;
    const uint32_t tP = tmem + lane_base + C::kColP;
    const float c = p.scale_log2;
    // A zero scale makes every visible score 0: use 0 as the score and 1 as
    // the multiplier.
    const bool zero_scale = !(c > 0.f);
    const float ce = zero_scale ? 1.f : c;
    // Bounded wait of all 32 lanes; a time-out is recorded once.
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      bool wv = ptx::mbar_wait(bar, parity, limit);
      wv = __all_sync(0xffffffffu, wv);
      if (!wv) fail();
      return wv;
    };

    bool ok = true;
    int n = 0;  // KV steps so far (global, across items)
    int u = 0;  // items with work so far
    for (int k = 0; ok; ++k) {
      const int item = qitem_at(k, n_items);
      if (item < 0) break;
      const QItem w = decode_qitem(p, item, num_qblocks);
      if (w.lo >= w.hi) continue;
      const int i = w.q0 + row;
      const RowBounds rb = row_bounds(p, i);

      float m_use = -INFINITY;  // running max of score * scale * log2(e) (possibly stale)
      float l_run = 0.f;        // running sum of 2^(x - m_use)
      for (int j = w.lo; j < w.hi; ++j, ++n) {
        if (!wait_all(bar_s_full, static_cast<uint32_t>(n) & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        rec(tr::kSReady, j);

        uint32_t r[kBN];
        float pm[kBN / 32];  // maximum of each 32 columns, reduced by the load
#pragma unroll
        for (int c0 = 0; c0 < kBN; c0 += 32)
          ptx::tmem_ld_max_32x32b_x32(tS + c0, r + c0, &pm[c0 / 32]);
        ptx::tmem_wait_ld();
        ptx::reg_fence<kBN>(r);
        tile::float_fence<kBN / 32>(pm);
        // S(n) is in registers: the next S may be computed over it.
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_s_free);
        rec(tr::kSLoaded, j);

        const int k0 = j * kBN;
        bool full = k0 + kBN <= p.S;
        if (p.causal) full = full && (k0 + kBN - 1 <= w.q0);
        if (p.window > 0) full = full && (w.q0 + kBM - 1 - k0 < p.window);
        if (p.window > 0 && !p.causal) full = full && (k0 + kBN - 1 - w.q0 < p.window);
        const int vlo = rb.lo == INT_MIN ? INT_MIN : rb.lo - k0;
        const int vhi = rb.hi - k0;

        // Tiles that straddle the mask boundary (or a zero scale): hide the
        // invisible scores in place, then every tile takes the same path.
        if (!full || zero_scale) tile::mask_cols(r, vlo, vhi, zero_scale);

        // Row maximum of the (visible) scores: from the loads' reductions
        // when every score is visible, else over the masked registers.
        float mx;
        if (full && !zero_scale)
          mx = tile::max_of(pm);
        else
          mx = tile::row_max(r);
        if (FA_TRACE) {
          asm volatile("" ::"f"(mx));
          rec(tr::kMaxDone, j);
        }
        const float m_tile = mx == -INFINITY ? -INFINITY : mx * ce;
        const float m_new = fmaxf(m_use, m_tile);
        const bool first = j == w.lo;
        float alpha = 1.f;
        bool rescale = false;
        if (first) {
          m_use = m_new;
        } else if (m_new > m_use + kRescaleThreshold) {
          alpha = ptx::ex2_approx(m_use - m_new);  // m_use may be -inf: alpha = 0
          m_use = m_new;
          rescale = true;
        }
        const float neg_base = m_use == -INFINITY ? 0.f : -m_use;

        // P = 2^(x - m_use) (hidden scores are -inf and give 0) as bf16
        // pairs, and the row sum.
        const float row_sum = tile::exp2_to_bf16(r, ce, neg_base);
        l_run = l_run * alpha + row_sum;
        if (FA_TRACE) {
          asm volatile("" ::"f"(l_run), "r"(r[0]), "r"(r[63]));
          rec(tr::kExpDone, j);
        }
        // PV(n - 1) reads P's columns and accumulates into O: it must have
        // completed before P is overwritten or O corrected.
        if (n > 0) {
          if (!wait_all(bar_pv_done, static_cast<uint32_t>(n - 1) & 1u)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
        }
#pragma unroll
        for (int c0 = 0; c0 < kBN / 2; c0 += 32) ptx::tmem_st_32x32b_x32(tP + c0, r + c0);

        // Lazy correction of the O accumulator.
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
        if (lane == 0) ptx::mbar_arrive(bar_p_full);
        rec(tr::kPReady, j | (rescale ? 1u << 23 : 0u));
      }

      // ---- epilogue: O -> registers (then O's columns go back to the MMA
      // thread) -> O / l as bf16 in shared memory, swizzled, over this item's
      // Q buffer (its S MMAs are done) -> TMA store; LSE. A warp that timed
      // out records it in misc[2] before the barrier, so the four warps leave
      // together.
      if (ok && !wait_all(bar_o_full, static_cast<uint32_t>(u) & 1u)) ok = false;
      if (!ok && lane == 0) misc[2] = 1;
      // A store of rows that start past S would be a planning error.
      const bool do_store = ok && tr::guard(w.q0 < p.S, p.status, kStatusBoundsGuard);
      const int qb = u & 1;
      if (do_store) {
        rec(tr::kEpilogueStart, 0);
        ptx::tc_fence_after();
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        uint8_t* stage = smem + C::kQOff + qb * C::kTileBytes;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          ptx::tmem_ld_32x32b_x32(tO + c0, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence<32>(o);
          tile::stage_bf16_sw128(stage, C::kBoxBytes, row, c0, o, inv_l);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_o_free);
      if (do_store) ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(1, 128);
      const bool failed = misc[2] != 0;
      if (warp == 0 && lane == 0) {
        if (!failed && do_store) {
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            ptx::tma_store_4d(&tm_o, sQ + qb * C::kTileBytes + bx * C::kBoxBytes, bx * C::kBoxCols,
                              w.h, w.q0, w.b);
          ptx::tma_store_commit();
          ptx::tma_store_wait_read();
        }
        // This Q buffer may take the item after next's Q.
        ptx::mbar_arrive(bar_q_free + 8 * qb);
      }
      if (failed) {
        ok = false;
        break;
      }
      if (do_store && p.lse != nullptr && i < p.S) {
        const float m_fin = m_use == -INFINITY ? 0.f : m_use;
        const long long idx = (static_cast<long long>(w.b) * p.H + w.h) * p.S + i;
        const long long lse_limit =
            p.lse_limit > 0 ? p.lse_limit : static_cast<long long>(p.B) * p.H * p.S;
        if (tr::guard(idx < lse_limit, p.status, kStatusBoundsGuard))
          p.lse[idx] = (m_fin + __log2f(l_run)) * kLn2;
      }
      if (do_store) rec(tr::kEpilogueEnd, 0);
      ++u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int QT>
cudaError_t launch_d(const FwdProblem& p, void* out, const void* q, const void* k, const void* v,
                     cudaStream_t stream) {
  using C = Cfg<D, QT>;
  CUtensorMap tq, tk, tv, to;
  // The maps carry the real head dim p.D <= D: loads zero-fill columns
  // p.D..D-1 (adding nothing to Q K^T and giving zero O columns) and the
  // store clips them.
  constexpr int bc = C::kBoxCols;
  if (!encode_bshd_tensor_map(&tq, q, p.B, p.S, p.H, p.D, p.sq, 1, kBM, p.cache_maps, bc) ||
      !encode_bshd_tensor_map(&tk, k, p.B, p.S, p.Hkv, p.D, p.sk, 1, kBN, p.cache_maps, bc) ||
      !encode_bshd_tensor_map(&tv, v, p.B, p.S, p.Hkv, p.D, p.sv, 1, kBN, p.cache_maps, bc) ||
      !encode_bshd_tensor_map(&to, out, p.B, p.S, p.H, p.D, p.so, 1, kBM, p.cache_maps, bc))
    return cudaErrorInvalidValue;
  const int nqb = (p.S + QT * kBM - 1) / (QT * kBM);
  const long long grid = static_cast<long long>(nqb) * p.H * p.B;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  // One-tile CTAs: the persistent kernel, with as many CTAs as there are
  // items or resident slots (not in the debug build, whose trace records one
  // item per CTA).
  if constexpr (QT == 1 && D == 64 && !FA_TRACE) {
    using PC = PCfg<D>;
    const long long ctas = std::min(grid, static_cast<long long>(p.num_sms) * PC::kCtasPerSm);
    if (p.num_sms > 0) {
      static unsigned long long attr_done = 0;
      cudaError_t err = ensure_smem_attr(
          &attr_done, reinterpret_cast<const void*>(&fa_fwd_bf16_tc_persistent_kernel<D>),
          PC::kSmemBytes);
      if (err != cudaSuccess) return err;
      fa_fwd_bf16_tc_persistent_kernel<D>
          <<<static_cast<unsigned>(ctas), PC::kThreads, PC::kSmemBytes, stream>>>(tq, tk, tv, to,
                                                                                   p, nqb);
      return cudaGetLastError();
    }
  }
  static unsigned long long attr_done = 0;
  cudaError_t err = ensure_smem_attr(&attr_done, reinterpret_cast<const void*>(
                                                     &fa_fwd_bf16_tc_kernel<D, QT>),
                                     C::kSmemBytes);
  if (err != cudaSuccess) return err;
  fa_fwd_bf16_tc_kernel<D, QT><<<static_cast<unsigned>(grid), Roles<QT>::kThreads, C::kSmemBytes,
                                 stream>>>(tq, tk, tv, to, p, nqb);
  return cudaGetLastError();
}

// Q tiles per CTA: one for head dims up to 64 -- a CTA of one tile fits
// twice on an SM and, run persistent with P in its own tensor-memory
// columns, computes S(j+1) during the softmax of j (B1 H16 S8192 D64 causal
// 786 -> 1005 TFLOP/s against two-tile CTAs; B4 H16 S1024: 280 -> 377) --
// else two (one CTA per SM; no tensor-memory room for P of its own).
int q_tiles_per_cta(int D, int S) {
  (void)S;
  return D <= 64 ? 1 : 2;
}

}  // namespace

int fwd_bf16_tc_ctas(int S, int D) {
  const int rows = q_tiles_per_cta(D, S) * kBM;
  return (S + rows - 1) / rows;
}

cudaError_t launch_fwd_bf16_tc(const FwdProblem& p, void* out, const void* q, const void* k,
                               const void* v, cudaStream_t stream) {
  // Head dims up to 64 (96, 128) run on the 64 (96, 128) column kernel.
  if (p.D % 8 != 0 || p.D < 8 || p.D > 128) return cudaErrorInvalidValue;
  if (p.D <= 64) return launch_d<64, 1>(p, out, q, k, v, stream);
  if (p.D <= 96) return launch_d<96, 2>(p, out, q, k, v, stream);
  return launch_d<128, 2>(p, out, q, k, v, stream);
}

}  // namespace fa
