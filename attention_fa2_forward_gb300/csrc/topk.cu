// topk.cu -- exact top-K selection per row (the op of the Modular recipe
// "Custom Operations: Applications in AI Models", section "Optimizing top-K
// token sampling for GPUs in MAX": each row of scores comes back ordered by
// highest value, as values and indices).
//
// Order: descending IEEE-754 total order (-NaN < -inf < ... < -0 < +0 < ...
// < +inf < +NaN); equal values by ascending index. Both rules are folded into
// one 64-bit key per element, larger = earlier in the output:
//   key = total_order_bits(x) << 32 | (0xffffffff - index)
// so the keys of one row are distinct and the answer is unique.
//
// The selection reads every score once from HBM and does a few instructions
// per element on the common path:
//   * chunk kernel: one CTA per (row chunk, batch); its 8 warps scan the
//     chunk interleaved (warp w takes every 8th block of 256 elements, so the
//     CTA streams one contiguous front of memory) without block barriers (8
//     elements per lane per step, staged by asynchronous 16-byte copies (4-byte
//     when the rows are not 16-byte aligned) in a shared-memory ring with
//     seven steps in flight). Before the scan the CTA seeds its threshold
//     from the first staged steps (all seven for a long chunk or a large K,
//     else four): the K-th largest of the per-lane, per-step maxima (1792 or
//     1024 distinct elements), rounded down, is a lower bound of the chunk's
//     K-th key. A
//     warp keeps only keys above the best threshold any warp of the CTA has
//     published (the value half of the key is compared first), each lane
//     appending its own rare candidates to a warp-private buffer;
//     when that buffer passes max(K, 256) keys the warp cuts it to its top K
//     with a radix select over the 64-bit keys (a byte per pass, stopping as
//     soon as the bucket holding the K-th key holds exactly the keys still
//     needed; warp-private histogram) and publishes its K-th key (the
//     smallest survivor) as a threshold for the whole CTA. At the end the CTA selects the top K of its warps'
//     survivors once (block-wide). A chunk that is the whole row writes
//     them sorted straight to the output; otherwise they go (padded with key
//     0, below every real key, when the chunk is shorter) to the workspace;
//   * rows of 2, 4 or 8 chunks with K <= 128: the row's chunk CTAs form a
//     thread-block cluster, and its first CTA reads the others' top K from
//     their shared memory, selects the row's top K and writes it;
//   * merge kernel (other multi-chunk rows): one CTA per row selects the top
//     K of the chunks' candidates the same way.
// Sorting K distinct keys: up to 128 each key's place is its count of
// larger keys, above that a bitonic sort.
// Scores are handled as raw 32-bit patterns from load to store: no float
// operation touches them, so NaN payloads and signed zeros survive.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "fa_internal.h"
#include "topk_plan.h"

namespace fa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = 8;                  // elements a lane reads per scan step
constexpr int kWarpStep = kPerThread * 32;     // elements a warp reads per scan step

__device__ __forceinline__ uint32_t total_order_bits(uint32_t b) {
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint64_t make_key(uint32_t bits, uint32_t index) {
  return (static_cast<uint64_t>(total_order_bits(bits)) << 32) | (0xffffffffu - index);
}

__device__ __forceinline__ uint32_t key_bits(uint64_t key) {
  const uint32_t t = static_cast<uint32_t>(key >> 32);
  return (t & 0x80000000u) ? (t & 0x7fffffffu) : ~t;
}

// Thread-block cluster helpers: this CTA's rank in its cluster, a barrier
// over every thread of the cluster (release / acquire: shared-memory writes
// before it are visible to the cluster's loads after it), and a load from a
// peer CTA's shared memory at the same offset as `local` (a shared-window
// address) in this CTA.
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}
__device__ __forceinline__ uint64_t ld_cluster_u64(uint32_t remote) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ int key_index(uint64_t key) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
}

struct SelectScratch {
  unsigned hist[256];
  int digit, k_rem, count;
};

// The K largest keys of a selection are exactly those with
// (key & mask) >= prefix.
struct Selection {
  uint64_t prefix, mask;
};

// Radix select of the top K of n keys in shared memory (K <= n; the K-th
// largest and everything above it distinct), most significant byte first:
// each pass histograms the byte of the keys still matching the prefix and a
// warp finds the byte holding the K-th. Stops once that byte's bucket holds
// exactly the keys still needed.
__device__ Selection block_select_top(const uint64_t* items, int n, int K, SelectScratch& sc) {
  uint64_t prefix = 0, mask = 0;
  int k_rem = K;
  const int tid = threadIdx.x;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kThreads) sc.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint64_t v = items[i];
      if ((v & mask) == prefix) atomicAdd(&sc.hist[(v >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // Lane l owns bytes 8l .. 8l+7; keys above lane l's bytes: the totals
      // of lanes l+1 .. 31.
      unsigned c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sc.hist[tid * 8 + j];
        tot += c[j];
      }
      unsigned incl = tot;  // inclusive suffix sum over lanes l .. 31
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned up = __shfl_down_sync(0xffffffffu, incl, o);
        if (tid + o < 32) incl += up;
      }
      const unsigned above = incl - tot;
      const unsigned kr = static_cast<unsigned>(k_rem);
      if (above < kr && kr <= incl) {
        unsigned cum = above;
        for (int j = 7; j >= 0; --j) {
          if (cum + c[j] >= kr) {
            sc.digit = tid * 8 + j;
            sc.k_rem = static_cast<int>(kr - cum);
            sc.count = static_cast<int>(c[j]);
            break;
          }
          cum += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= static_cast<uint64_t>(sc.digit) << shift;
    mask |= 0xffull << shift;
    k_rem = sc.k_rem;
    const bool done = sc.count == k_rem;  // every key left in the bucket is needed
    __syncthreads();                      // sc is rewritten by the next pass
    if (done) break;
  }
  return Selection{prefix, mask};
}

// The same radix select by one warp over its private keys, with its own
// histogram (no block barrier).
__device__ Selection warp_select_top(const uint64_t* items, int n, int K, unsigned* hist) {
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0, mask = 0;
  unsigned k_rem = static_cast<unsigned>(K);
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      const uint64_t v = items[i];
      if ((v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 255u], 1u);
    }
    __syncwarp();
    unsigned c[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[lane * 8 + j];
      tot += c[j];
    }
    unsigned incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned up = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += up;
    }
    const unsigned above = incl - tot;
    const bool found = above < k_rem && k_rem <= incl;
    int my_digit = 0;
    unsigned my_rem = 0, my_cnt = 0;
    if (found) {
      unsigned cum = above;
      for (int j = 7; j >= 0; --j) {
        if (cum + c[j] >= k_rem) {
          my_digit = lane * 8 + j;
          my_rem = k_rem - cum;
          my_cnt = c[j];
          break;
        }
        cum += c[j];
      }
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, found)) - 1;
    const int digit = __shfl_sync(0xffffffffu, my_digit, src);
    k_rem = __shfl_sync(0xffffffffu, my_rem, src);
    const unsigned cnt = __shfl_sync(0xffffffffu, my_cnt, src);
    prefix |= static_cast<uint64_t>(digit) << shift;
    mask |= 0xffull << shift;
    __syncwarp();
    if (cnt == k_rem) break;
  }
  return Selection{prefix, mask};
}

// Keeps the selected keys of a warp-private buffer, in place (each 32-key
// group is read before any write reaches it); returns their count.
__device__ int warp_compact(uint64_t* items, int n, Selection sel) {
  const int lane = threadIdx.x & 31;
  int w = 0;
  for (int r = 0; r < n; r += 32) {
    const int i = r + lane;
    const uint64_t v = i < n ? items[i] : 0ull;
    const bool keep = i < n && (v & sel.mask) >= sel.prefix;
    const unsigned ballot = __ballot_sync(0xffffffffu, keep);
    __syncwarp();
    if (keep) items[w + __popc(ballot & ((1u << lane) - 1u))] = v;
    w += __popc(ballot);
    __syncwarp();
  }
  return w;
}

// One scan step of a lane covers elements base + 4 * lane + {0..3} and
// base + 128 + 4 * lane + {0..3} (coalesced 16-byte groups across the warp).
// They are staged in the warp's ring of shared-memory slots by asynchronous
// copies (cp.async, L2 only), so the loads in flight hold no registers; a
// lane only reads back the words it copied itself. kVec: rows 16-byte
// aligned and V a multiple of 4 (16-byte copies); otherwise 4-byte copies.
// Words past the chunk end are zero-filled and masked by the filter.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool kVec>
__device__ __forceinline__ void stage_step(const uint32_t* row, int base, int end, uint32_t slot) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < kPerThread / 4; ++u) {
    const int i0 = base + 128 * u + 4 * lane;
    const uint32_t dst = slot + static_cast<uint32_t>((128 * u + 4 * lane) * 4);
    if (kVec) {
      const int bytes = i0 < end ? 16 : 0;
      cp_async_16(dst, bytes ? static_cast<const void*>(row + i0) : static_cast<const void*>(row),
                  bytes);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int bytes = i0 + e < end ? 4 : 0;
        cp_async_4(dst + 4 * e,
                   bytes ? static_cast<const void*>(row + i0 + e) : static_cast<const void*>(row),
                   bytes);
      }
    }
  }
  cp_async_commit();
}

__device__ __forceinline__ void read_step(const uint32_t* slot, uint32_t (&x)[kPerThread]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < kPerThread / 4; ++u) {
    const uint4 v = *reinterpret_cast<const uint4*>(slot + 128 * u + 4 * lane);
    x[4 * u] = v.x;
    x[4 * u + 1] = v.y;
    x[4 * u + 2] = v.z;
    x[4 * u + 3] = v.w;
  }
}

__device__ __forceinline__ int step_index(int base, int e) {
  return base + 128 * (e >> 2) + 4 * (static_cast<int>(threadIdx.x) & 31) + (e & 3);
}

// A warp's scan state: its private buffer (capacity cap = prune_at + one
// step), key count and threshold (both warp-uniform registers).
struct WarpScan {
  uint64_t* buf;
  unsigned* hist;
  int n, prune_at;           // key count (warp-uniform) and the prune trigger
  uint64_t thr;
  unsigned long long* best;  // the CTA's best threshold (shared memory)
  uint64_t best_seen;        // its value read one step ahead
};

__device__ __forceinline__ void filter_step(const uint32_t (&x)[kPerThread],
                                            const uint32_t* words, int base, int end, int K,
                                            WarpScan& ws) {
  const int lane = threadIdx.x & 31;
  // Common path, 2 to 4 integer operations per element: the value half of the
  // key as a signed integer in total order (b ^ ((b >> 31) & 0x7fffffff))
  // against the threshold's value half, conservatively (>=); the few elements
  // that pass get the exact 64-bit test below. Only a chunk's last blocks
  // need the bounds test.
  // Any warp's K-th key is a lower bound of the CTA's K-th key: filter
  // against the best one published so far, read during the previous step so
  // that its latency stays off this step's path.
  ws.thr = max(ws.thr, ws.best_seen);
  ws.best_seen = *reinterpret_cast<volatile unsigned long long*>(ws.best);
  const int32_t s_thr = static_cast<int32_t>(static_cast<uint32_t>(ws.thr >> 32) ^ 0x80000000u);
  unsigned mask = 0;
  if (base + kWarpStep <= end && s_thr >= 0) {
    // A threshold value >= +0 (the usual case once seeded): raw bits compare
    // as signed integers directly, negative scores and -NaN being negative
    // integers below it.
#pragma unroll
    for (int e = 0; e < kPerThread; ++e)
      if (static_cast<int32_t>(x[e]) >= s_thr) mask |= 1u << e;
  } else if (base + kWarpStep <= end) {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int32_t v = static_cast<int32_t>(x[e]);
      if ((v ^ ((v >> 31) & 0x7fffffff)) >= s_thr) mask |= 1u << e;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int32_t v = static_cast<int32_t>(x[e]);
      if (step_index(base, e) < end && (v ^ ((v >> 31) & 0x7fffffff)) >= s_thr) mask |= 1u << e;
    }
  }
  // Candidates are rare (the threshold starts seeded): a step without any
  // costs one vote. Otherwise the warp takes one set bit per lane per round:
  // the value comes back from this step's staging slot (intact until the
  // next step), and a ballot gives each taken key its place after the warp's
  // count (no atomics, the count stays in a register).
  if (!__any_sync(0xffffffffu, mask != 0)) return;
  const unsigned below = (1u << lane) - 1u;
  do {
    bool take = false;
    uint64_t key = 0;
    if (mask != 0) {
      const int e = __ffs(mask) - 1;
      mask &= mask - 1;
      const uint32_t v = words[128 * (e >> 2) + 4 * lane + (e & 3)];
      key = make_key(v, static_cast<uint32_t>(step_index(base, e)));
      take = key > ws.thr;
    }
    const unsigned taken = __ballot_sync(0xffffffffu, take);
    if (take) ws.buf[ws.n + __popc(taken & below)] = key;
    ws.n += __popc(taken);
  } while (__any_sync(0xffffffffu, mask != 0));
  if (ws.n > ws.prune_at) {
    __syncwarp();
    const Selection sel = warp_select_top(ws.buf, ws.n, K, ws.hist);
    ws.n = warp_compact(ws.buf, ws.n, sel);
    __syncwarp();
    // The new threshold is the exact K-th key, the smallest survivor (the
    // selection may stop at a coarse bucket; its floor would let many keys
    // through): later keys must beat it to matter.
    uint64_t m = ~0ull;
    for (int i = lane; i < ws.n; i += 32) m = min(m, ws.buf[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (ws.n >= K) {  // a K-th key exists: publish it
      ws.thr = m;
      if (lane == 0) atomicMax(ws.best, static_cast<unsigned long long>(m));
    }
  }
}

// Writes K distinct keys (shared memory, room for P >= K entries, P the next
// power of two; every thread of the CTA calls this after a barrier) to one
// output row in descending order. Up to kRankSortMax keys each key's place
// is the number of larger keys (no barriers, K reads per key); above that a
// bitonic sort over P entries padded with key 0.
constexpr int kRankSortMax = 128;
__device__ void write_sorted_row(uint64_t* keys, int K, uint32_t* values, int* indices) {
  if (K <= kRankSortMax) {
    for (int i = threadIdx.x; i < K; i += kThreads) {
      const uint64_t v = keys[i];
      int r = 0;
      for (int j = 0; j < K; ++j) r += keys[j] > v ? 1 : 0;
      values[r] = key_bits(v);
      indices[r] = key_index(v);
    }
    return;
  }
  int P = 1;
  while (P < K) P <<= 1;
  for (int i = K + threadIdx.x; i < P; i += kThreads) keys[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P / 2; i += kThreads) {
        const int lo = 2 * i - (i & (stride - 1));  // pairs (lo, lo + stride)
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = keys[lo], c = keys[hi];
        if ((a < c) == desc) {
          keys[lo] = c;
          keys[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < K; i += kThreads) {
    values[i] = key_bits(keys[i]);
    indices[i] = key_index(keys[i]);
  }
}

// Dynamic shared memory of the chunk kernel: per warp a ring of kRing
// staging slots (kWarpStep words each), a key buffer of prune_at + kWarpStep
// keys and a 256-bin histogram, then the CTA's merge area of kWarps * K keys.
constexpr int kRing = 8;
// Scan steps per warp that seed the threshold: all the prologue stages for a
// long chunk or a large K, fewer for a short chunk, whose few steps cannot
// amortise waiting for the last staged one.
constexpr int kSeedStepsLong = kRing - 1;
constexpr int kSeedStepsShort = 4;
static_assert(kSeedStepsShort * kThreads >= kMaxTopK, "at least K groups seed the threshold");
static_assert(kSeedStepsLong * kThreads <= kWarps * 2 * kWarpStep, "seed keys fit the key buffers");
constexpr int kRingKeys = kWarps * kRing * kWarpStep / 2;  // 64-bit keys the ring holds
static_assert(kWarps * kMaxTopK <= kRingKeys, "the warps' top K always fit the idle ring");
static_assert(kWarps >= 2, "the merge area (kWarps * K keys) holds the sort buffer");
__host__ __device__ inline int chunk_prune_at(int K) { return K > 256 ? K : 256; }
__host__ __device__ inline size_t chunk_smem_bytes(int K) {
  return static_cast<size_t>(kWarps) * kRing * kWarpStep * sizeof(uint32_t) +
         static_cast<size_t>(kWarps) * (chunk_prune_at(K) + kWarpStep) * sizeof(uint64_t) +
         static_cast<size_t>(kWarps) * 256 * sizeof(unsigned) +
         static_cast<size_t>(kWarps) * K * sizeof(uint64_t);
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    topk_chunk_kernel(const float* __restrict__ scores, long long row_stride, int V, int K,
                      int chunk, int n_chunks, uint64_t* __restrict__ cand,
                      uint32_t* __restrict__ values, int* __restrict__ indices, int clustered) {
  extern __shared__ uint64_t dyn[];
  __shared__ SelectScratch sc;
  __shared__ int s_count[kWarps];
  __shared__ unsigned long long s_best;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int b = blockIdx.y;
  const int prune_at = chunk_prune_at(K);
  const int wcap = prune_at + kWarpStep;
  uint32_t* rings = reinterpret_cast<uint32_t*>(dyn);
  uint64_t* wbufs = reinterpret_cast<uint64_t*>(rings + kWarps * kRing * kWarpStep);
  unsigned* hists = reinterpret_cast<unsigned*>(wbufs + kWarps * wcap);
  uint64_t* merged = reinterpret_cast<uint64_t*>(hists + kWarps * 256);

  // The warps interleave over the chunk: at step s warp w takes block
  // ((s + rot) mod steps) * 8 + w of kWarpStep elements, so the CTA reads one
  // contiguous front of memory (8 blocks per step, kRing - 1 steps ahead).
  // The rotation rot differs between CTAs: chunks start at multiples of the
  // chunk size, and CTAs walking them in lockstep would hit the same address
  // bits (the same L2 slices and memory channels) at the same time.
  const int start = c * chunk;
  const int cend = min(V, start + chunk);
  const int nblocks = (cend - start + kWarpStep - 1) / kWarpStep;
  const int steps = (nblocks + kWarps - 1) / kWarps;
  const int rot = static_cast<int>((static_cast<unsigned>(b) * 2654435761u +
                                    static_cast<unsigned>(c) * 40503u) %
                                   static_cast<unsigned>(steps > 0 ? steps : 1));
  auto block_base = [&](int s) {  // s < 2 * steps
    int r = s + rot;
    if (r >= steps) r -= steps;
    return start + (r * kWarps + warp) * kWarpStep;
  };
  const uint32_t* row =
      reinterpret_cast<const uint32_t*>(scores) + static_cast<long long>(b) * row_stride;
  if (threadIdx.x == 0) s_best = 0ull;
  __syncthreads();
  WarpScan ws{wbufs + warp * wcap, hists + warp * 256, 0, prune_at, 0ull, &s_best, 0ull};

  // kRing - 1 steps in flight: at step s the copy of step s + kRing - 1 goes
  // into the slot step s - 1 used, then the oldest copy group is awaited.
  uint32_t* ring = rings + warp * kRing * kWarpStep;
  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  // Steps past the last one stage nothing (zero-byte copies) but still
  // commit a group, which keeps the group count uniform.
  auto stage = [&](int s, int slot_i) {
    stage_step<kVec>(row, s < steps ? block_base(s) : cend, cend,
                     ring_s + slot_i * kWarpStep * 4);
  };
#pragma unroll
  for (int r = 0; r < kRing - 1; ++r) stage(r, r);

  // Seed the CTA's threshold from the first seed_steps steps of every warp
  // (already staged): per lane and step the largest of its scores, one
  // distinct element per group, as a key whose low half is a distinct id
  // (key 0 marks a group without elements). The value half of the K-th
  // largest of these keys, rounded down by the radix select, is at or below
  // at least K elements of the chunk, so it bounds the chunk's K-th key from
  // below: nothing the top K needs is filtered out. Starting every warp near
  // the K-th of the 8 * seed_steps * kThreads sampled scores instead of from
  // zero leaves a warp with a few dozen candidates per chunk and rarely a
  // prune.
  const bool long_seed = steps >= 32 || K > 256;  // uniform over the CTA
  const int seed_steps = long_seed ? kSeedStepsLong : kSeedStepsShort;
  if (long_seed)
    cp_async_wait<kRing - 1 - kSeedStepsLong>();
  else
    cp_async_wait<kRing - 1 - kSeedStepsShort>();
#pragma unroll
  for (int s = 0; s < kSeedStepsLong; ++s) {
    if (s >= seed_steps) break;
    uint32_t x[kPerThread];
    read_step(ring + s * kWarpStep, x);
    int32_t best = INT_MIN;
    bool any = false;
    if (s < steps) {
      const int base = block_base(s);
#pragma unroll
      for (int e = 0; e < kPerThread; ++e) {
        const int32_t v = static_cast<int32_t>(x[e]);
        if (step_index(base, e) < cend) {
          best = max(best, v ^ ((v >> 31) & 0x7fffffff));
          any = true;
        }
      }
    }
    const uint32_t id = static_cast<uint32_t>(s * kThreads + threadIdx.x);
    wbufs[id] = any ? (static_cast<uint64_t>(static_cast<uint32_t>(best) ^ 0x80000000u) << 32) |
                          (id + 1u)
                    : 0ull;
  }
  __syncthreads();
  {
    const Selection seed = block_select_top(wbufs, seed_steps * kThreads, K, sc);
    if (threadIdx.x == 0) s_best = seed.prefix & 0xffffffff00000000ull;
  }
  __syncthreads();  // the key buffers are reused by the scan
  ws.thr = ws.best_seen = s_best;

  int slot = 0;
  for (int st = 0; st < steps; ++st) {
    const int next = slot == 0 ? kRing - 1 : slot - 1;
    stage(st + kRing - 1, next);
    cp_async_wait<kRing - 1>();
    uint32_t x[kPerThread];
    read_step(ring + slot * kWarpStep, x);
    filter_step(x, ring + slot * kWarpStep, block_base(st), cend, K, ws);  // past cend: masked
    slot = slot == kRing - 1 ? 0 : slot + 1;
  }
  cp_async_wait<0>();
  __syncwarp();
  if (lane == 0) s_count[warp] = ws.n;
  __syncthreads();
  // The warps' keys are gathered into the staging ring, idle now that every
  // copy has landed, and the CTA selects its top K once. Only when they would
  // not fit (large K) does each warp first cut its own keys to K.
  int total = 0;
  for (int w = 0; w < kWarps; ++w) total += s_count[w];
  if (total > kRingKeys) {
    if (ws.n > K) {
      const Selection sel = warp_select_top(ws.buf, ws.n, K, ws.hist);
      ws.n = warp_compact(ws.buf, ws.n, sel);
    }
    __syncthreads();  // every warp has read the old counts
    if (lane == 0) s_count[warp] = ws.n;
    __syncthreads();
    total = 0;
    for (int w = 0; w < kWarps; ++w) total += s_count[w];
  }
  int off = 0;
  for (int w = 0; w < warp; ++w) off += s_count[w];
  uint64_t* gathered = reinterpret_cast<uint64_t*>(rings);
  for (int i = lane; i < ws.n; i += 32) gathered[off + i] = ws.buf[i];
  __syncthreads();
  // The CTA's top K go to the merge area: the keys are distinct, so exactly
  // K match the selection (the bound only keeps a broken invariant inside
  // the K slots).
  uint64_t* top = merged;
  if (total > K) {
    const Selection sel = block_select_top(gathered, total, K, sc);
    if (threadIdx.x == 0) sc.count = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const uint64_t v = gathered[i];
      if ((v & sel.mask) >= sel.prefix) {
        const int slot = atomicAdd(&sc.count, 1);
        if (slot < K) top[slot] = v;
      }
    }
  } else {
    for (int i = threadIdx.x; i < K; i += kThreads) top[i] = i < total ? gathered[i] : 0ull;
  }
  __syncthreads();
  if (n_chunks == 1) {  // the chunk is the whole row: its top K is the answer
    write_sorted_row(top, K, values + static_cast<long long>(b) * K,
                     indices + static_cast<long long>(b) * K);
  } else if (clustered) {
    // The row's chunk CTAs form one cluster (rank = chunk): rank 0 reads the
    // others' top K from their shared memory, selects the row's top K and
    // writes it. The keys of a row are distinct and every chunk gave
    // min(K, its length) real keys, so the K largest are real; padding keys
    // (0) sort below them.
    cluster_sync();  // every chunk's top K is in its shared memory
    if (cluster_rank() == 0) {
      const int n = n_chunks * K;  // <= kRingKeys
      uint64_t* gathered = reinterpret_cast<uint64_t*>(rings);
      const uint32_t top_s = static_cast<uint32_t>(__cvta_generic_to_shared(top));
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int r = i / K, e = i - r * K;
        gathered[i] = r == 0 ? top[e] : ld_cluster_u64(cluster_map(top_s + 8u * e, r));
      }
      __syncthreads();
      const Selection sel = block_select_top(gathered, n, K, sc);
      if (threadIdx.x == 0) sc.count = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint64_t v = gathered[i];
        if ((v & sel.mask) >= sel.prefix) {
          const int slot = atomicAdd(&sc.count, 1);  // < K while the invariant holds
          if (slot < K) top[slot] = v;
        }
      }
      __syncthreads();
      write_sorted_row(top, K, values + static_cast<long long>(b) * K,
                       indices + static_cast<long long>(b) * K);
    }
    cluster_sync();  // no CTA leaves while rank 0 may still read its shared memory
  } else {
    uint64_t* dst = cand + (static_cast<long long>(b) * n_chunks + c) * K;
    for (int i = threadIdx.x; i < K; i += kThreads) dst[i] = top[i];
  }
}

__global__ void __launch_bounds__(kThreads)
    topk_merge_kernel(const uint64_t* __restrict__ cand, int n_chunks, int K,
                      uint32_t* __restrict__ values, int* __restrict__ indices) {
  extern __shared__ uint64_t items[];  // n_chunks * K candidates, then the sort buffer
  __shared__ SelectScratch sc;
  const int b = blockIdx.x;
  const int n = n_chunks * K;
  const uint64_t* src = cand + static_cast<long long>(b) * n;
  for (int i = threadIdx.x; i < n; i += kThreads) items[i] = src[i];
  __syncthreads();
  // The padding keys (0) repeat, but the K largest are real and distinct:
  // every chunk contributed min(K, its length) real keys and V >= K.
  const Selection top = block_select_top(items, n, K, sc);
  // The K winners into the sort buffer (room for P >= K keys after the
  // candidates), then out in order.
  uint64_t* sel = items + n;
  if (threadIdx.x == 0) sc.count = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kThreads)
    if ((items[i] & top.mask) >= top.prefix) {
      const int slot = atomicAdd(&sc.count, 1);  // < K while the invariant holds
      if (slot < K) sel[slot] = items[i];
    }
  __syncthreads();
  write_sorted_row(sel, K, values + static_cast<long long>(b) * K,
                   indices + static_cast<long long>(b) * K);
}

}  // namespace

cudaError_t launch_topk(const TopkProblem& p, cudaStream_t stream) {
  if (p.B < 1 || p.V < 1 || p.K < 1 || p.K > kMaxTopK || p.n_chunks < 1 ||
      static_cast<long long>(p.n_chunks) * p.K > kMaxTopkCandidates || p.B > 65535)
    return cudaErrorInvalidValue;
  const bool vec = reinterpret_cast<uintptr_t>(p.scores) % 16 == 0 && p.row_stride % 4 == 0 &&
                   p.V % 4 == 0;
  if (p.chunk % (kWarps * kWarpStep) != 0) return cudaErrorInvalidValue;
  const size_t csmem = chunk_smem_bytes(p.K);
  const bool clustered = topk_clustered(p.n_chunks, p.K) && p.n_chunks > 1;
  static_assert(2 * (kWarps * kRing * kWarpStep * sizeof(uint32_t) +
                     kWarps * (256 + kWarpStep) * sizeof(uint64_t) +
                     kWarps * 256 * sizeof(unsigned) + kWarps * kTopkClusterMaxK * sizeof(uint64_t) +
                     2048) <= 228 * 1024,
                "two chunk CTAs share an SM up to the largest clustered K");
  static_assert(kTopkMaxCluster * kMaxTopK <= kRingKeys, "a cluster's candidates fit the ring");
  static_assert(kWarps * kRing * kWarpStep * 4 + kWarps * (kMaxTopK + kWarpStep) * 8 +
                        kWarps * 256 * 4 + kWarps * kMaxTopK * 8 <= 227 * 1024,
                "the largest K's chunk CTA fits the shared-memory limit");
  // Each kernel's shared-memory limit is raised once per device, to what the
  // largest K needs.
  static unsigned long long attr_done[2] = {0, 0};
  auto launch = [&](auto kernel, int which) -> cudaError_t {
    cudaError_t e = ensure_smem_attr(&attr_done[which], reinterpret_cast<const void*>(kernel),
                                     static_cast<int>(chunk_smem_bytes(kMaxTopK)));
    if (e != cudaSuccess) return e;
    uint32_t* vals = reinterpret_cast<uint32_t*>(p.values);
    if (!clustered) {
      kernel<<<dim3(p.n_chunks, p.B), kThreads, csmem, stream>>>(
          p.scores, p.row_stride, p.V, p.K, p.chunk, p.n_chunks, p.cand, vals, p.indices, 0);
      return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_chunks, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = csmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.n_chunks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p.scores, p.row_stride, p.V, p.K, p.chunk,
                              p.n_chunks, p.cand, vals, p.indices, 1);
  };
  cudaError_t err = vec ? launch(topk_chunk_kernel<true>, 1) : launch(topk_chunk_kernel<false>, 0);
  if (err != cudaSuccess) return err;
  err = cudaGetLastError();
  if (err != cudaSuccess || p.n_chunks == 1 || clustered) return err;  // rows already finished
  int P = 1;
  while (P < p.K) P <<= 1;
  const size_t smem = (static_cast<size_t>(p.n_chunks) * p.K + P) * sizeof(uint64_t);
  static unsigned long long merge_attr_done = 0;
  err = ensure_smem_attr(&merge_attr_done, reinterpret_cast<const void*>(&topk_merge_kernel),
                         static_cast<int>((kMaxTopkCandidates + kMaxTopK) * sizeof(uint64_t)));
  if (err != cudaSuccess) return err;
  topk_merge_kernel<<<p.B, kThreads, smem, stream>>>(
      p.cand, p.n_chunks, p.K, reinterpret_cast<uint32_t*>(p.values), p.indices);
  return cudaGetLastError();
}

}  // namespace fa
