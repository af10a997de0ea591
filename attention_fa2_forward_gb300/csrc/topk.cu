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
//     seven steps in flight). A
//     warp keeps only keys above the best threshold any warp of the CTA has
//     published (the value half of the key is compared first), each lane
//     appending its own rare candidates to a warp-private buffer;
//     when that buffer passes max(K, 256) keys the warp cuts it to its top K
//     with a radix select over the 64-bit keys (a byte per pass, stopping as
//     soon as the bucket holding the K-th key holds exactly the keys still
//     needed; warp-private histogram) and publishes its K-th key (the
//     smallest survivor) as a threshold for the whole CTA. At the end the CTA selects the top K of its warps'
//     survivors once (block-wide) and writes them (padded with key 0, below
//     every real key, when the chunk is shorter) to the workspace;
//   * merge kernel: one CTA per row selects the top K of the chunks'
//     candidates the same way and sorts them (bitonic, descending).
// Scores are handled as raw 32-bit patterns from load to store: no float
// operation touches them, so NaN payloads and signed zeros survive.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "fa_internal.h"

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
  int n, prune_at;
  uint64_t thr;
  unsigned long long* best;  // the CTA's best threshold (shared memory)
  int* count;                // the warp's key count (shared memory; n mirrors it)
};

__device__ __forceinline__ void filter_step(const uint32_t (&x)[kPerThread], int base, int end,
                                            int K, WarpScan& ws) {
  const int lane = threadIdx.x & 31;
  // Common path, 4 integer operations per element: the value half of the key
  // as a signed integer in total order (b ^ ((b >> 31) & 0x7fffffff)) against
  // the threshold's value half, conservatively (>=); the few elements that
  // pass get the exact 64-bit test below. Only a chunk's last blocks need the
  // bounds test.
  // Any warp's K-th key is a lower bound of the CTA's K-th key: filter
  // against the best one published so far.
  ws.thr = max(ws.thr, static_cast<uint64_t>(*reinterpret_cast<volatile unsigned long long*>(
                           ws.best)));
  const int32_t s_thr = static_cast<int32_t>(static_cast<uint32_t>(ws.thr >> 32) ^ 0x80000000u);
  unsigned mask = 0;
  if (base + kWarpStep <= end) {
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
  // Candidates are rare: each lane appends its own, taking slots from the
  // warp's counter in shared memory (no per-element warp votes).
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    if ((mask >> e) & 1u) {
      const uint64_t key = make_key(x[e], static_cast<uint32_t>(step_index(base, e)));
      if (key > ws.thr) ws.buf[atomicAdd(ws.count, 1)] = key;
    }
  }
  __syncwarp();
  ws.n = *reinterpret_cast<volatile int*>(ws.count);
  if (ws.n > ws.prune_at) {
    __syncwarp();
    const Selection sel = warp_select_top(ws.buf, ws.n, K, ws.hist);
    ws.n = warp_compact(ws.buf, ws.n, sel);
    if (lane == 0) *ws.count = ws.n;
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

// Dynamic shared memory of the chunk kernel: per warp a ring of kRing
// staging slots (kWarpStep words each), a key buffer of prune_at + kWarpStep
// keys and a 256-bin histogram, then the CTA's merge area of kWarps * K keys.
constexpr int kRing = 8;
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
                      int chunk, int n_chunks, uint64_t* __restrict__ cand) {
  extern __shared__ uint64_t dyn[];
  __shared__ SelectScratch sc;
  __shared__ int s_count[kWarps];
  __shared__ unsigned long long s_best;
  __shared__ int s_wcount[kWarps];
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
  if (lane == 0) s_wcount[warp] = 0;
  __syncthreads();
  WarpScan ws{wbufs + warp * wcap, hists + warp * 256, 0, prune_at, 0ull, &s_best,
              &s_wcount[warp]};

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
  int slot = 0;
  for (int st = 0; st < steps; ++st) {
    const int next = slot == 0 ? kRing - 1 : slot - 1;
    stage(st + kRing - 1, next);
    cp_async_wait<kRing - 1>();
    uint32_t x[kPerThread];
    read_step(ring + slot * kWarpStep, x);
    filter_step(x, block_base(st), cend, K, ws);  // blocks past cend are masked out
    slot = slot == kRing - 1 ? 0 : slot + 1;
  }
  cp_async_wait<0>();
  __syncwarp();
  if (ws.n > K) {
    const Selection sel = warp_select_top(ws.buf, ws.n, K, ws.hist);
    ws.n = warp_compact(ws.buf, ws.n, sel);
  }
  if (lane == 0) s_count[warp] = ws.n;
  __syncthreads();
  // Gather the warps' survivors (at most K each) and select the CTA's top K.
  int off = 0, total = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) off += s_count[w];
    total += s_count[w];
  }
  for (int i = lane; i < ws.n; i += 32) merged[off + i] = ws.buf[i];
  __syncthreads();
  uint64_t* dst = cand + (static_cast<long long>(b) * n_chunks + c) * K;
  if (total > K) {
    const Selection sel = block_select_top(merged, total, K, sc);
    if (threadIdx.x == 0) sc.count = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const uint64_t v = merged[i];
      if ((v & sel.mask) >= sel.prefix) dst[atomicAdd(&sc.count, 1)] = v;
    }
  } else {
    for (int i = threadIdx.x; i < K; i += kThreads) dst[i] = i < total ? merged[i] : 0ull;
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
  // The K winners into the sort buffer (P = next power of two >= K, padded
  // with 0), then a bitonic sort into descending order.
  int P = 1;
  while (P < K) P <<= 1;
  uint64_t* sel = items + n;
  for (int i = threadIdx.x; i < P; i += kThreads) sel[i] = 0ull;
  if (threadIdx.x == 0) sc.count = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kThreads)
    if ((items[i] & top.mask) >= top.prefix) sel[atomicAdd(&sc.count, 1)] = items[i];
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P / 2; i += kThreads) {
        const int lo = 2 * i - (i & (stride - 1));  // pairs (lo, lo + stride)
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = sel[lo], c = sel[hi];
        if ((a < c) == desc) {
          sel[lo] = c;
          sel[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < K; i += kThreads) {
    values[static_cast<long long>(b) * K + i] = key_bits(sel[i]);
    indices[static_cast<long long>(b) * K + i] = key_index(sel[i]);
  }
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
  cudaError_t err;
  if (vec) {
    err = cudaFuncSetAttribute(topk_chunk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(csmem));
    if (err != cudaSuccess) return err;
    topk_chunk_kernel<true><<<dim3(p.n_chunks, p.B), kThreads, csmem, stream>>>(
        p.scores, p.row_stride, p.V, p.K, p.chunk, p.n_chunks, p.cand);
  } else {
    err = cudaFuncSetAttribute(topk_chunk_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(csmem));
    if (err != cudaSuccess) return err;
    topk_chunk_kernel<false><<<dim3(p.n_chunks, p.B), kThreads, csmem, stream>>>(
        p.scores, p.row_stride, p.V, p.K, p.chunk, p.n_chunks, p.cand);
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  int P = 1;
  while (P < p.K) P <<= 1;
  const size_t smem = (static_cast<size_t>(p.n_chunks) * p.K + P) * sizeof(uint64_t);
  err = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  topk_merge_kernel<<<p.B, kThreads, smem, stream>>>(
      p.cand, p.n_chunks, p.K, reinterpret_cast<uint32_t*>(p.values), p.indices);
  return cudaGetLastError();
}

}  // namespace fa
