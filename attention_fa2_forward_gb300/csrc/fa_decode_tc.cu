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
//   * a unit is one (KV head, position tile, batch); an item is a range of
//     its KV tiles streamed through a shared-memory ring. When the units
//     fill the GPU, every CTA runs one unit whole. Otherwise persistent CTAs
//     share the work -- stream-K: groups of Hkv CTAs (one per KV head, all
//     reading the same cache rows) take equal contiguous quotas of all the
//     position-tile groups' KV tiles, found from the lengths on the device;
//     or, on request, fixed splits of every unit taken round-robin -- and
//     carry their pipeline from one item to the next (ring, S buffers, two Q
//     and two O buffers). Each piece of a cut unit writes its partial result
//     (O / l in fp32 and the LSE) to a slot; a second kernel merges a unit's
//     slots with weights exp(LSE_piece - LSE);
//   * S is double-buffered in tensor memory (S_0, S_1 at columns 0 and 128,
//     O at 256 and 256 + D): the MMA warp computes S(j+1) while the softmax
//     warps work on S(j). The issue order is S0 S1 | PV0 S2 | PV1 S3 | ...;
//     an item's epilogue runs after the next item's first P is stored;
//   * only the softmax warps whose tensor-memory lanes hold real rows work;
//   * V rows of an item's last tile that lie past L_b but inside the cache are
//     zeroed in shared memory by the softmax warps before they release the
//     step's P to the PV MMA (their P is 0, but 0 * NaN would not be).
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
constexpr uint32_t kColO = 256;          // O buffer o at columns [256 + o * D, 256 + (o + 1) * D)
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr unsigned long long kDrainExtraNs = 100000000ull;  // 100 ms

// One item: a range of KV tiles of one (KV head, position tile, batch) unit,
// and the slot its partial result goes to (split modes).
struct Item {
  int hk, pt, b;
  int L, sq0, nq, pos0;
  int jlo, jhi, n;   // KV tiles [jlo, jhi), n = jhi - jlo
  int piece;         // partial-result slot (split modes)
  bool v_fix;        // the last tile holds cache rows past L_b
};

// KV tiles [t0, t1) the unit (hk, pt, b) needs (empty: t0 == t1), and the
// rows' geometry; the same for every KV head.
struct UnitRange {
  int L, sq0, nq, pos0, t0, t1;
};

// Keys of batch b (clamped into [0, Scache]).
__device__ __forceinline__ int batch_len(const DecodeProblem& p, int b) {
  return min(max(p.lens != nullptr ? p.lens[b] : p.Scache, 0), p.Scache);
}

__device__ __forceinline__ UnitRange unit_range_of(const DecodeProblem& p, int pt, int L) {
  UnitRange u;
  u.L = L;
  u.sq0 = pt * p.Pq;              // first query row of the tile
  u.nq = min(p.Pq, p.Sq - u.sq0);  // query positions in the tile
  u.pos0 = u.L - p.Sq + u.sq0;     // position of the first of them
  const int posl = u.pos0 + u.nq - 1;
  // Keys any row of the tile may see: [klo, khi].
  const int klo = p.window > 0 ? max(0, u.pos0 - p.window + 1) : 0;
  const int khi = p.causal ? min(posl, u.L - 1)
                           : (p.window > 0 ? min(posl + p.window - 1, u.L - 1) : u.L - 1);
  u.t0 = u.t1 = 0;
  if (khi >= klo) {
    u.t0 = klo / kBN;
    u.t1 = khi / kBN + 1;
  }
  return u;
}

__device__ __forceinline__ UnitRange unit_range(const DecodeProblem& p, int pt, int b) {
  return unit_range_of(p, pt, batch_len(p, b));
}

// Units are numbered (position-tile group, KV head) with the KV head fastest:
// group grp = (batch b, position tile pt, latest first -- under the causal
// mask later position tiles see more keys), unit = grp * Hkv + hk. CTAs that
// run together then read the same cache rows of every KV head (whole rows of
// [.., Hkv, D]).
__device__ __forceinline__ int group_pt(const DecodeProblem& p, int grp) {
  return p.n_ptiles - 1 - grp % p.n_ptiles;
}

__device__ __forceinline__ Item make_item(const DecodeProblem& p, const UnitRange& u, int hk,
                                          int pt, int b, int jlo, int jhi, int piece) {
  Item it;
  it.hk = hk;
  it.pt = pt;
  it.b = b;
  it.L = u.L;
  it.sq0 = u.sq0;
  it.nq = u.nq;
  it.pos0 = u.pos0;
  it.jlo = jlo;
  it.jhi = jhi;
  it.n = jhi - jlo;
  it.piece = piece;
  it.v_fix = it.n > 0 && (it.L % kBN) != 0 && it.L < p.Scache && it.jhi - 1 == it.L / kBN;
  return it;
}

// Stream-K mode: the CTA groups (Hkv consecutive CTAs, one per KV head)
// share the position-tile groups' KV tiles laid end to end (W in total) in
// equal contiguous quotas of q >= stream_k_min tiles; the Hkv CTAs of a group
// read the same cache rows, each for its own KV head.
__device__ __forceinline__ long long stream_k_quota(const DecodeProblem& p, long long w) {
  const long long cg = p.persistent / p.Hkv;  // CTA groups
  long long q = (w + cg - 1) / cg;
  return q < p.stream_k_min ? p.stream_k_min : q;
}

// Quotas that group tiles [P, P + T) touch: the pieces each of its units is
// cut into.
__device__ __forceinline__ long long unit_pieces(long long P, long long T, long long q) {
  return T > 0 ? (P + T - 1) / q - P / q + 1 : 0;
}

// One entry of a CTA's item list: unit, KV tiles [jlo, jhi), partial slot,
// and the batch's key count (so that no role reads the lengths again).
struct ItemRef {
  int unit, jlo, jhi, piece, L;
};
constexpr int kMaxItems = kDecodeMaxItems;  // list capacity (the plan sizes the work to fit)

__device__ __forceinline__ Item load_item(const DecodeProblem& p, const ItemRef& r) {
  const int hk = r.unit % p.Hkv;
  const int grp = r.unit / p.Hkv;
  const int pt = group_pt(p, grp);
  const int b = grp / p.n_ptiles;
  return make_item(p, unit_range_of(p, pt, r.L), hk, pt, b, r.jlo, r.jhi, r.piece);
}

// The items of this CTA, in order (lane 0 of warp 0 builds the list; the
// other lanes return 0):
//   grid mode: unit blockIdx.x, whole (also without keys: its rows get O = 0);
//   fixed splits: every gridDim.x-th of the units' `splits` ranges that hold
//     keys, slot unit * splits + split;
//   stream-K: for each group overlapping this CTA group's quota [lo, hi), the
//     overlap for this CTA's KV head; slot base * Hkv + hk * pieces + k, with
//     base = the pieces of the groups before, k = this quota's index among
//     those the group touches.
// (A warp-parallel version of this list, lane per group, measured 12 %
// slower on fixed splits although it built the same lists.)
__device__ __noinline__ int build_items(const DecodeProblem& p, ItemRef* list, int lane) {
  if (lane != 0) return 0;
  const int g = static_cast<int>(blockIdx.x);
  if (p.persistent == 0) {
    const int grp = g / p.Hkv;
    const int L = batch_len(p, grp / p.n_ptiles);
    const UnitRange u = unit_range_of(p, group_pt(p, grp), L);
    list[0] = ItemRef{g, u.t0, u.t1, 0, L};
    return 1;
  }
  const int groups = p.n_ptiles * p.B;
  int count = 0;
  if (p.stream_k_min == 0) {
    const long long C = gridDim.x;
    long long i = g;
    for (int grp = 0; grp < groups && count < kMaxItems; ++grp) {
      const int L = batch_len(p, grp / p.n_ptiles);
      const UnitRange u = unit_range_of(p, group_pt(p, grp), L);
      const long long ns = (u.t1 - u.t0 + p.tiles_per_split - 1) / p.tiles_per_split;
      const long long nk = ns * p.Hkv;
      for (; i < nk && count < kMaxItems; i += C) {
        const int split = static_cast<int>(i / p.Hkv);
        const int hk = static_cast<int>(i % p.Hkv);
        const int jlo = u.t0 + split * p.tiles_per_split;
        const int unit = grp * p.Hkv + hk;
        list[count++] = ItemRef{unit, jlo, min(u.t1, jlo + p.tiles_per_split),
                                unit * p.splits + split, L};
      }
      i -= nk;
    }
    return count;
  }
  long long w = 0;
  for (int grp = 0; grp < groups; ++grp) {
    const UnitRange u = unit_range(p, group_pt(p, grp), grp / p.n_ptiles);
    w += u.t1 - u.t0;
  }
  const long long q = stream_k_quota(p, w);
  const int hk = g % p.Hkv;
  const long long lo = static_cast<long long>(g / p.Hkv) * q, hi = lo + q;
  long long P = 0, base = 0;
  for (int grp = 0; grp < groups && P < hi && count < kMaxItems; ++grp) {
    const int L = batch_len(p, grp / p.n_ptiles);
    const UnitRange u = unit_range_of(p, group_pt(p, grp), L);
    const long long T = u.t1 - u.t0;
    const long long a = lo > P ? lo : P;
    const long long e = hi < P + T ? hi : P + T;
    const long long pieces = unit_pieces(P, T, q);
    if (e > a) {
      const long long k = g / p.Hkv - P / q;
      list[count++] = ItemRef{grp * p.Hkv + hk, u.t0 + static_cast<int>(a - P),
                              u.t0 + static_cast<int>(e - P),
                              static_cast<int>(base * p.Hkv + hk * pieces + k), L};
    }
    base += pieces;
    P += T;
  }
  return count;
}

template <int D>
struct DCfg {
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  // Q area: two Q buffers, so that the next item's Q loads while this item's
  // last S MMAs read the current one. At D = 128 and 256 the area holds one
  // 128-row tile: two buffers of 64 rows when the tile has at most 64 real
  // rows (MMA rows 64..127 then read whatever follows in shared memory; they
  // belong to no softmax warp and are never read back), else one buffer.
  static constexpr int kQArea = D == 64 ? 2 * kTileBytes : kTileBytes;
  // Ring slots: what fits next to the Q area in 227 KB. Two slots suffice for
  // the ring order (K0 K1 | V0 K2 | ...): each refill waits only on an MMA
  // that needs nothing later in the ring.
  static constexpr int kStages = D == 256 ? 2 : (D == 128 ? 6 : 11);
  // O buffers in tensor memory (after S_0, S_1): two let an item's epilogue
  // run while the next item accumulates into the other.
  static constexpr int kOBufs = D == 256 ? 1 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQArea;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2] pv_done
  // o_full[2] o_empty[2] drain epi
  static constexpr int kNumBars = 4 + 2 * kStages + 2 + 2 + 1 + 4 + 1 + 1;
  // The CTA's item list, then the misc words.
  static constexpr int kItemOff = (kBarOff + kNumBars * 8 + 15) & ~15;
  static constexpr int kMiscOff = kItemOff + kMaxItems * static_cast<int>(sizeof(ItemRef)) + 16;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack for 1 KB alignment
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(256 + kOBufs * D <= static_cast<int>(kTmemCols), "tensor memory");
  static_assert(kQArea >= kTileBytes, "the unsplit epilogue stages O over the Q area");
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
  const uint32_t bar_q_full = bars;                               // + 8 qbuf
  const uint32_t bar_q_empty = bars + 16;                         // + 8 qbuf
  const uint32_t bar_kv_full = bars + 32;                         // + 8 s
  const uint32_t bar_kv_empty = bar_kv_full + 8 * C::kStages;     // + 8 s
  const uint32_t bar_s_full = bar_kv_empty + 8 * C::kStages;      // + 8 buf
  const uint32_t bar_p_full = bar_s_full + 16;                    // + 8 buf
  const uint32_t bar_pv_done = bar_p_full + 16;
  const uint32_t bar_o_full = bar_pv_done + 8;                    // + 8 obuf
  const uint32_t bar_o_empty = bar_o_full + 16;                   // + 8 obuf
  const uint32_t bar_drain = bar_o_empty + 16;
  const uint32_t bar_epi = bar_drain + 8;  // the softmax warps' epilogue stores are done
  ItemRef* items = reinterpret_cast<ItemRef*>(smem + C::kItemOff);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
  // misc[0]: tensor-memory base address, misc[1]: abort flag, misc[2]: items

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nact = (p.R + 31) >> 5;       // softmax warps holding real rows
  // Q buffers and their layout: qbufs buffers of kBoxes boxes, q_box bytes
  // (q_box / 128 rows of 128 bytes) per box.
  const int qbufs = (D == 64 || p.R <= 64) ? 2 : 1;
  const int q_box = C::kQArea / (qbufs * C::kBoxes);
  const int q_buf = q_box * C::kBoxes;
  const unsigned long long limit = p.wait_limit_ns;
  const unsigned long long drain_limit = limit + kDrainExtraNs;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar_q_full + 8 * t, 1);
      ptx::mbar_init(bar_q_empty + 8 * t, 1);
      ptx::mbar_init(bar_s_full + 8 * t, 1);
      ptx::mbar_init(bar_p_full + 8 * t, nact);
      ptx::mbar_init(bar_o_full + 8 * t, 1);
      ptx::mbar_init(bar_o_empty + 8 * t, nact);
    }
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar_kv_full + 8 * s, 1);
      ptx::mbar_init(bar_kv_empty + 8 * s, 1);
    }
    ptx::mbar_init(bar_pv_done, 1);
    ptx::mbar_init(bar_drain, 1);
    ptx::mbar_init(bar_epi, nact);
    misc[1] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    const int n = build_items(p, items, lane);
    if (lane == 0) misc[2] = static_cast<uint32_t>(n);
  }
  // Rows R.. of each Q box are never loaded: zero them once so that the MMA
  // rows of the softmax warps' lanes past R read defined values (their
  // results are never stored).
  {
    const int zrow_bytes = q_box - p.R * 128;
    const int chunks = zrow_bytes >> 4;  // 16-byte chunks per box
    for (int e = threadIdx.x; e < qbufs * C::kBoxes * chunks; e += kThreads) {
      const int bx = e / chunks;  // box over all buffers
      const int off = (e % chunks) << 4;
      *reinterpret_cast<uint4*>(smem + C::kQOff + bx * q_box + p.R * 128 + off) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    ptx::fence_proxy_async_smem();
  }
  // The combine kernel (launched as a programmatic dependent) may start
  // loading: it waits for this grid to finish before it reads the results.
  if (threadIdx.x == 0) ptx::launch_dependents();
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
  const int nitems = static_cast<int>(misc[2]);

  auto fail = [&]() {
    misc[1] = 1;
    atomicOr(p.status, kStatusWaitTimeout);
  };
  auto aborted = [&]() { return misc[1] != 0; };

  if (warp == kLoadWarp) {
    // ===================================================== TMA producer
    if (lane == 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      // A single position tile streams the cache once; several (prefill, or
      // long query chunks) read each K/V tile again: keep those in L2.
      const uint64_t pol_kv =
          p.n_ptiles > 1 ? ptx::policy_evict_last() : ptx::policy_evict_first();
      uint32_t armed = 0, armed_parity = 0;  // per slot: loaded at least once / last parity
      int idx = 0, kw = 0;                   // ring entries, items with keys so far
      bool ok = true;
      for (int it = 0; ok && it < nitems; ++it) {
        const Item I = load_item(p, items[it]);
        if (I.n == 0) continue;
        const int qs = kw % qbufs;
        // The Q buffer is free once the S MMAs of the item that used it last
        // have completed.
        if (kw >= qbufs &&
            (aborted() || !ptx::mbar_wait(bar_q_empty + 8 * qs,
                                          static_cast<uint32_t>((kw - qbufs) / qbufs) & 1u,
                                          limit))) {
          fail();
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(bar_q_full + 8 * qs, C::kBoxes * p.R * 128);
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          ptx::tma_load_4d(sQ + qs * q_buf + bx * q_box, &tm_q, bar_q_full + 8 * qs, bx * 64,
                           I.hk * p.G, I.sq0, I.b, pol_q);
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
                             bx * 64, I.hk, j * kBN, I.b, pol_kv);
          armed |= 1u << s;
          armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
        };
        // Ring order = MMA consumption order: K0 K1 | V0 K2 | V1 K3 | ...
        issue(0, I.jlo);
        if (ok && I.n > 1) issue(0, I.jlo + 1);
        for (int r = 0; r < I.n && ok; ++r) {
          issue(1, I.jlo + r);
          if (ok && r + 2 < I.n) issue(0, I.jlo + r + 2);
        }
        ++kw;  // counts the Q loads issued
      }
      // Never leave while a copy of ours may still be writing shared memory.
      for (int qb = 0; qb < qbufs && qb < kw; ++qb) {
        const int loads = (kw - qb + qbufs - 1) / qbufs;  // Q loads into buffer qb
        ptx::mbar_wait(bar_q_full + 8 * qb, static_cast<uint32_t>(loads - 1) & 1u, drain_limit);
      }
      for (int s = 0; s < C::kStages; ++s)
        if ((armed >> s) & 1u)
          ptx::mbar_wait(bar_kv_full + 8 * s, (armed_parity >> s) & 1u, drain_limit);
    }
  } else if (warp == kMmaWarp) {
    // ===================================================== MMA issuer (lane 0)
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, D, false, true);
    bool ok = true;
    // Test hook: wait on the drain barrier, which nothing signals before
    // this warp's own final commit, so the bounded wait must expire.
    if (p.stall_probe) {
      bool w = lane == 0 ? ptx::mbar_wait(bar_drain, 0, limit) : true;
      if (!__shfl_sync(0xffffffffu, w, 0)) {
        if (lane == 0) fail();
        ok = false;
      }
    }
    int idx = 0, R = 0, kw = 0;  // ring entries, S/PV steps, items with keys so far
    const uint64_t dk0 = ptx::smem_desc_sw128(sKV, 16, 1024);
    const uint64_t dv0 = ptx::smem_desc_sw128(sKV, kBoxBytes, 1024);
    // Waits for phase `parity` of `bar`.
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
      bool w = !aborted() && ptx::mbar_wait(bar, parity, limit);
      if (!w) fail();
      if (w) ptx::tc_fence_after();
      return w;
    };
    auto wait_kv = [&]() -> int {
      const int s = idx % C::kStages;
      const uint32_t ph = static_cast<uint32_t>(idx / C::kStages) & 1u;
      ++idx;
      return wait(bar_kv_full + 8 * s, ph) ? s : -1;
    };
    for (int it = 0; lane == 0 && ok && it < nitems; ++it) {
      const Item I = load_item(p, items[it]);
      const int n = I.n;
      if (n == 0) continue;
      const int qs = kw % qbufs;
      const int ob = kw % C::kOBufs;
      const uint32_t tO = tmem + kColO + static_cast<uint32_t>(ob * D);
      ok = wait(bar_q_full + 8 * qs, static_cast<uint32_t>(kw / qbufs) & 1u);
      if (!ok) break;
      const uint64_t dq = ptx::smem_desc_sw128(sQ + qs * q_buf, 16, 1024);
      auto issue_s = [&](int buf, int kslot, bool last_s) {
        const uint64_t dk = dk0 + static_cast<uint32_t>((kslot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offq = static_cast<uint32_t>(((kk >> 2) * q_box + (kk & 3) * 32) >> 4);
          const uint32_t offk = static_cast<uint32_t>(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          ptx::mma_ss(tmem + buf * kBN, dq + offq, dk + offk, kIdescS, kk > 0 ? 1u : 0u);
        }
        ptx::tc_commit(bar_s_full + 8 * buf);
        ptx::tc_commit(bar_kv_empty + 8 * kslot);
        if (last_s) ptx::tc_commit(bar_q_empty + 8 * qs);  // Q is read by S MMAs only
      };
      auto issue_pv = [&](int buf, int vslot, bool accumulate) {
        const uint64_t dv = dv0 + static_cast<uint32_t>((vslot * C::kTileBytes) >> 4);
        const uint32_t acc = accumulate ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          ptx::mma_ts(tO, tmem + buf * kBN + kk * 8, dv + static_cast<uint32_t>(kk * 128),
                      kIdescPV, kk > 0 ? 1u : acc);
        ptx::tc_commit(bar_pv_done);
        ptx::tc_commit(bar_kv_empty + 8 * vslot);
      };

      {
        const int ks = wait_kv();
        ok = ks >= 0;
        if (!ok) break;
        issue_s(R & 1, ks, n == 1);
      }
      if (n > 1) {
        const int ks = wait_kv();
        ok = ks >= 0;
        if (!ok) break;
        issue_s((R + 1) & 1, ks, n == 2);
      }
      for (int r = 0; ok && r < n; ++r) {
        const int buf = (R + r) & 1;
        const int vs = wait_kv();
        ok = vs >= 0;
        if (!ok) break;
        // The first PV of an item overwrites its O buffer: the softmax warps
        // must have read the result of the item that used it before.
        if (r == 0 && kw >= C::kOBufs) {
          ok = wait(bar_o_empty + 8 * ob, static_cast<uint32_t>((kw - C::kOBufs) / C::kOBufs) & 1u);
          if (!ok) break;
        }
        ok = wait(bar_p_full + 8 * buf, static_cast<uint32_t>((R + r) >> 1) & 1u);
        if (!ok) break;
        issue_pv(buf, vs, r > 0);
        if (r + 2 < n) {
          const int ks = wait_kv();
          ok = ks >= 0;
          if (!ok) break;
          issue_s(buf, ks, r + 2 == n - 1);
        }
      }
      if (!ok) break;
      ptx::tc_commit(bar_o_full + 8 * ob);
      R += n;
      ++kw;
    }
    // Every MMA must have finished before tensor memory is released.
    if (lane == 0) {
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
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const float c = p.scale_log2;
    const bool zero_scale = !(c > 0.f);
    const float ce = zero_scale ? 1.f : c;

    // Partial result of a split item: O / l (fp32) and its LSE, once the
    // item's O buffer `ob` is final (its completion number ekw / kOBufs on
    // o_full[ob]). The tensor-memory loads are warp-collective (.sync.aligned):
    // every lane issues them; only real rows store.
    // Partial result of a piece: O / l (fp32) and its LSE to row `row` of
    // slot `piece`, once the item's O buffer is final (its completion number
    // ekw / kOBufs on o_full[ob]). The tensor-memory loads are warp-collective
    // (.sync.aligned): every lane issues them; only real rows store.
    auto split_epilogue = [&](bool valid, int piece, float l_run, float m_use, int ekw) -> bool {
      const int ob = ekw % C::kOBufs;
      const uint32_t tO = tmem + lane_base + kColO + static_cast<uint32_t>(ob * D);
      bool w = ptx::mbar_wait(bar_o_full + 8 * ob, static_cast<uint32_t>(ekw / C::kOBufs) & 1u,
                              limit);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        fail();
        return false;
      }
      ptx::tc_fence_after();
      const size_t prow = static_cast<size_t>(piece) * p.R + row;
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      if (valid)
        p.lse_part[prow] = l_run > 0.f
                               ? ((m_use == -INFINITY ? 0.f : m_use) + __log2f(l_run)) * kLn2
                               : -INFINITY;
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
      // O has been read: a later item's first PV may overwrite it.
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_o_empty + 8 * ob);
      return true;
    };
    // With two O buffers a split item's epilogue waits until the next item's
    // first P is stored, so that it runs while the tensor cores work.
    const bool defer = p.persistent > 0 && C::kOBufs == 2;
    bool pending = false, pend_valid = false;
    int pend_piece = 0, pend_kw = 0;
    float pend_l = 0.f, pend_m = 0.f;

    int R = 0, kw = 0, ring = 0;  // S/PV steps, items with keys, ring entries so far
    bool ok = true;
    for (int it = 0; ok && it < nitems; ++it) {
      const Item I = load_item(p, items[it]);
      const int n = I.n;
      const bool valid = row < p.R && pq < I.nq;
      const int sq = I.sq0 + pq;
      const int h = I.hk * p.G + g;
      const int pos = I.pos0 + pq;
      const uint32_t tO =
          tmem + lane_base + kColO + static_cast<uint32_t>((kw % C::kOBufs) * D);
      // Visible keys of this row: [vlo, vhi] (absolute positions).
      const int vlo = p.window > 0 ? max(pos - p.window + 1, 0) : 0;
      const int vhi = p.causal ? min(pos, I.L - 1)
                               : (p.window > 0 ? min(pos + p.window - 1, I.L - 1) : I.L - 1);

      float m_use = -INFINITY;  // running max of score * scale * log2(e) (possibly stale)
      float l_run = 0.f;        // running sum of 2^(x - m_use)
      for (int r = 0; r < n; ++r) {
        const int buf = (R + r) & 1;
        const uint32_t tS = tmem + lane_base + buf * kBN;
        bool w = ptx::mbar_wait(bar_s_full + 8 * buf, static_cast<uint32_t>((R + r) >> 1) & 1u,
                                limit);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          fail();
          ok = false;
          break;
        }
        ptx::tc_fence_after();

        uint32_t s[kBN];
        float pm[kBN / 32];  // maximum of each 32 columns, reduced by the load
#pragma unroll
        for (int c0 = 0; c0 < kBN; c0 += 32) ptx::tmem_ld_max_32x32b_x32(tS + c0, s + c0, &pm[c0 / 32]);
        ptx::tmem_wait_ld();
        ptx::reg_fence<kBN>(s);
        tile::float_fence<kBN / 32>(pm);

        // Rows that are not real (padding) are never stored: skip their mask.
        const int k0 = (I.jlo + r) * kBN;
        const bool full = !valid || (vlo <= k0 && k0 + kBN - 1 <= vhi);
        if (!full || zero_scale)
          tile::mask_cols(s, valid ? vlo - k0 : 0, valid ? vhi - k0 : kBN - 1, zero_scale);

        // Row maximum: from the loads' reductions when no score is hidden.
        float mx;
        if (full && !zero_scale)
          mx = tile::max_of(pm);
        else
          mx = tile::row_max(s);
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

        // Lazy correction of O: PV(R + r - 1) must have completed first (S of
        // this step was issued before it, so the S barrier does not imply
        // that).
        if (__any_sync(0xffffffffu, rescale)) {
          bool wp = ptx::mbar_wait(bar_pv_done, static_cast<uint32_t>(R + r - 1) & 1u, limit);
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
        if (r == n - 1 && I.v_fix) {
          // V rows of the last tile past L_b (inside the cache) may hold
          // anything; their P is 0, but 0 * NaN is not: zero them before the
          // PV MMA reads them (it waits for this P). V(n - 1) is the item's
          // last ring entry; every thread waits for it so that its stores
          // follow the copy.
          const int e = ring + 2 * n - 1;
          const int vs = e % C::kStages;
          bool wv = ptx::mbar_wait(bar_kv_full + 8 * vs,
                                   static_cast<uint32_t>(e / C::kStages) & 1u, limit);
          wv = __all_sync(0xffffffffu, wv);
          if (!wv) {
            fail();
            ok = false;
            break;
          }
          const int r0 = I.L - (I.jhi - 1) * kBN;                 // first row past L_b
          const int r1 = min(kBN, p.Scache - (I.jhi - 1) * kBN);  // rows the copy filled
          const int chunks = (r1 - r0) * 8;                        // 16-byte chunks per box
          uint8_t* vt = smem + C::kKVOff + vs * C::kTileBytes + r0 * 128;
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            for (int c16 = row; c16 < chunks; c16 += 32 * nact)
              *reinterpret_cast<uint4*>(vt + bx * kBoxBytes + c16 * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          ptx::fence_proxy_async_smem();
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_p_full + 8 * buf);
        if (r == 0 && pending) {
          pending = false;
          if (!split_epilogue(pend_valid, pend_piece, pend_l, pend_m, pend_kw)) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) break;

      // ---- epilogue of the item
      if (p.persistent > 0) {
        if (defer) {
          pending = true;
          pend_valid = valid;
          pend_piece = I.piece;
          pend_l = l_run;
          pend_m = m_use;
          pend_kw = kw;
        } else if (!split_epilogue(valid, I.piece, l_run, m_use, kw)) {
          ok = false;
          break;
        }
      } else {
        // O / l -> bf16 -> shared (swizzled, over the Q area) -> TMA store.
        // One item per CTA: the Q area is free once O is final.
        const bool has_o = n > 0;
        if (has_o) {
          bool w = ptx::mbar_wait(bar_o_full, 0, limit);
          w = __all_sync(0xffffffffu, w);
          if (!w) {
            fail();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
        }
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
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
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_epi);
        // Every softmax warp has staged its rows (bounded wait): store.
        if (warp == 0 && lane == 0) {
          if (ptx::mbar_wait(bar_epi, 0, limit)) {
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
              ptx::tma_store_4d(&tm_o, sQ + bx * kBoxBytes, bx * 64, I.hk * p.G, I.sq0, I.b);
            ptx::tma_store_commit();
            ptx::tma_store_wait_read();
          } else {
            fail();
          }
        }
        if (valid && p.lse != nullptr)
          p.lse[(static_cast<size_t>(I.b) * p.H + h) * p.Sq + sq] =
              l_run > 0.f ? ((m_use == -INFINITY ? 0.f : m_use) + __log2f(l_run)) * kLn2
                          : -INFINITY;
      }
      if (n > 0) {
        R += n;
        ++kw;
        ring += 2 * n;
      }
    }
    if (ok && pending) split_epilogue(pend_valid, pend_piece, pend_l, pend_m, pend_kw);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Merges the pieces' partial results: one CTA per unit (KV head, position
// tile, batch); warp 0 finds the unit's slots [first, first + ns) before the
// dependency wait (launched as a programmatic dependent of the attention
// kernel, it may run that part while the attention kernel still works: the
// lengths are not written there), then each warp merges whole rows of the
// unit's Q tile, loading several pieces at once. Partial rows hold D (padded)
// floats; out rows hold the real p.D <= D. O = sum_i w_i O_i / sum_i w_i and
// LSE = M + ln(sum_i w_i), with w_i = exp(LSE_i - M), M = max_i LSE_i; pieces
// whose row saw no key (LSE_i = -inf) are skipped, and a row no piece saw
// gets O = 0, LSE = -inf.
constexpr int kCombineWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32, 4)
    fa_decode_combine_kernel(const DecodeProblem p, __nv_bfloat16* __restrict__ out) {
  constexpr int kPer = D / 32;
  constexpr int kUnroll = D == 256 ? 4 : 8;  // pieces in flight per warp
  __shared__ long long sh_first, sh_ns;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int unit = static_cast<int>(blockIdx.x);
  const int hk = unit % p.Hkv;
  const int grp = unit / p.Hkv;
  const int pt = group_pt(p, grp);
  const int b = grp / p.n_ptiles;
  const int sq0 = pt * p.Pq;
  const int rows = min(p.Pq, p.Sq - sq0) * p.G;  // real rows of the unit's Q tile
  if (warp == 0) {
    if (p.stream_k_min > 0) {
      // The quota (all groups' tiles) and, for this group, the tiles and
      // pieces of the groups before it: 32 groups at a time (lane scans).
      const int groups = p.n_ptiles * p.B;
      auto tiles = [&](int g2) -> long long {
        if (g2 >= groups) return 0;
        const UnitRange u = unit_range(p, group_pt(p, g2), g2 / p.n_ptiles);
        return u.t1 - u.t0;
      };
      long long w = 0;
      for (int g0 = 0; g0 < groups; g0 += 32) w += tiles(g0 + lane);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
      const long long q = stream_k_quota(p, w);
      long long P = 0, base = 0;  // tiles and pieces of the groups before the chunk
      for (int g0 = 0; g0 <= grp; g0 += 32) {
        const long long T = tiles(g0 + lane);
        long long tp = T;  // inclusive scan of the tiles
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long v = __shfl_up_sync(0xffffffffu, tp, o);
          if (lane >= o) tp += v;
        }
        const long long pc = unit_pieces(P + tp - T, T, q);
        long long pp = pc;  // inclusive scan of the pieces
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long v = __shfl_up_sync(0xffffffffu, pp, o);
          if (lane >= o) pp += v;
        }
        if (g0 + lane == grp) {
          sh_first = (base + pp - pc) * p.Hkv + static_cast<long long>(hk) * pc;
          sh_ns = pc;
        }
        P += __shfl_sync(0xffffffffu, tp, 31);
        base += __shfl_sync(0xffffffffu, pp, 31);
      }
    } else if (lane == 0) {
      const UnitRange u = unit_range(p, pt, b);
      sh_first = static_cast<long long>(unit) * p.splits;
      sh_ns = (u.t1 - u.t0 + p.tiles_per_split - 1) / p.tiles_per_split;
    }
  }
  __syncthreads();
  const long long first = sh_first, ns = sh_ns;
  ptx::grid_dependency_wait();

  const size_t o_stride = static_cast<size_t>(p.R) * D;  // between slots
  for (int r = warp; r < rows; r += kCombineWarps) {
    // Slot s of row r: lse at (first + s) * R + r, O row at that times D.
    const float* lse_row = p.lse_part + static_cast<size_t>(first) * p.R + r;
    const float* o_row = p.o_part + (static_cast<size_t>(first) * p.R + r) * D + lane * kPer;
    float m = -INFINITY, wsum = 0.f;  // running max, weights and weighted O relative to it
    float acc[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) acc[u] = 0.f;
    for (long long s0 = 0; s0 < ns; s0 += kUnroll) {
      float ls[kUnroll];
      float x[kUnroll][kPer];
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const long long s = s0 + t;
        ls[t] = -INFINITY;
#pragma unroll
        for (int u = 0; u < kPer; ++u) x[t][u] = 0.f;
        if (s < ns) {
          ls[t] = lse_row[s * p.R];
          const float* src = o_row + s * o_stride;
          if constexpr (kPer % 4 == 0) {
#pragma unroll
            for (int u = 0; u < kPer; u += 4) {
              const float4 v = *reinterpret_cast<const float4*>(src + u);
              x[t][u] = v.x;
              x[t][u + 1] = v.y;
              x[t][u + 2] = v.z;
              x[t][u + 3] = v.w;
            }
          } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            x[t][0] = v.x;
            x[t][1] = v.y;
          }
        }
      }
      float m_new = m;
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) m_new = fmaxf(m_new, ls[t]);
      if (m_new == -INFINITY) continue;
      if (m != -INFINITY && m_new > m) {
        const float c = expf(m - m_new);
        wsum *= c;
#pragma unroll
        for (int u = 0; u < kPer; ++u) acc[u] *= c;
      }
      m = m_new;
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        if (ls[t] == -INFINITY) continue;  // no key for this row, or past ns
        const float w = expf(ls[t] - m);
        wsum += w;
#pragma unroll
        for (int u = 0; u < kPer; ++u) acc[u] = fmaf(w, x[t][u], acc[u]);
      }
    }
    const int sq = sq0 + r / p.G;
    const int h = hk * p.G + r % p.G;
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16* dst = out + static_cast<size_t>(b) * p.so.b +
                         static_cast<size_t>(sq) * p.so.s + static_cast<size_t>(h) * p.so.h +
                         lane * kPer;
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
      p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + sq] =
          wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
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
  const long long grid =
      p.persistent > 0 ? p.persistent : static_cast<long long>(p.Hkv) * p.n_ptiles * p.B;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  static unsigned long long attr_done = 0;
  cudaError_t err = ensure_smem_attr(&attr_done, reinterpret_cast<const void*>(
                                                     &fa_decode_bf16_tc_kernel<D>),
                                     DCfg<D>::kSmemBytes);
  if (err != cudaSuccess) return err;
  fa_decode_bf16_tc_kernel<D><<<static_cast<unsigned>(grid), kThreads, DCfg<D>::kSmemBytes,
                                stream>>>(tq, tk, tv, to, p);
  err = cudaGetLastError();
  if (err != cudaSuccess || p.persistent == 0) return err;
  const long long units = static_cast<long long>(p.Hkv) * p.n_ptiles * p.B;
  if (units > INT_MAX) return cudaErrorInvalidConfiguration;
  DecodeProblem pc = p;  // the combine kernel addresses out with resolved strides
  pc.so = resolve_strides(p.so, p.Sq, p.H, p.D);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units));
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D>, pc,
                            static_cast<__nv_bfloat16*>(out));
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
