// fa_internal.h -- declarations shared by the host C-ABI and the kernels'
// launchers (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

// Bits of the status word the kernels may set.
constexpr unsigned kStatusWaitTimeout = 1u;
constexpr unsigned kStatusBoundsGuard = 2u;  // debug build: a bounds guard skipped an access

// Element strides of a BSHD (or BShD) view along B, S and H; D is
// contiguous. All zero means the dense layout of the view's shape.
struct BshdStrides {
  long long b = 0, s = 0, h = 0;
};

// The dense strides when `st` is all zero, else `st`.
inline BshdStrides resolve_strides(BshdStrides st, int S, int heads, int D) {
  if (st.b == 0 && st.s == 0 && st.h == 0) {
    st.h = D;
    st.s = static_cast<long long>(heads) * D;
    st.b = static_cast<long long>(S) * heads * D;
  }
  return st;
}

// Problem description handed to both kernels by value.
struct FwdProblem {
  int B, S, H, Hkv, D;
  int causal;            // 1: key j visible to query i only if j <= i
  int window;            // > 0: also require i - j < window
  float scale;           // multiplies q.k
  float scale_log2;      // scale * log2(e)
  float* lse;            // [B, H, S] fp32 or nullptr
  unsigned* status;      // device status word (sticky error bits)
  unsigned long long wait_limit_ns;
  int stall_probe;       // test hook: the MMA issuer first waits on a barrier nothing signals
  BshdStrides sq, sk, sv, so;  // layouts of q, k, v, out (zero: dense)
  void* trace = nullptr;       // debug build: event records (fa_trace.cuh), or nullptr
  long long trace_ctas = 0;    // CTAs the trace buffer has room for
  long long lse_limit = 0;     // debug build: LSE elements a guard lets the kernel write
  bool cache_maps = true;      // false: encode the tensor maps without the (allocating) cache
  int num_sms = 0;             // > 0: the device's SMs; the bf16 kernel may then run persistent
};

// Attention over a KV cache (bf16, tensor cores): batch b holds L_b keys at
// the start of a [B, Scache, Hkv, D] cache; its Sq queries ([B, Sq, H, D])
// sit at positions L_b - Sq .. L_b - 1. A Q tile packs Pq positions x G heads
// of one KV head (R = G * Pq <= 128 rows); a unit is one (b, KV head,
// position tile). Three ways to share out the units' KV tiles:
//   persistent = 0: a CTA per unit, each unit whole (no partial results);
//   persistent = C > 0, stream_k_min = 0: C CTAs; each unit is cut into
//     `splits` ranges of `tiles_per_split` tiles and the CTAs take every C-th
//     of the ranges that hold keys;
//   persistent = C > 0, stream_k_min > 0: C CTAs take equal contiguous
//     quotas (at least stream_k_min tiles) of all units' tiles laid end to
//     end, found from the lengths on the device.
// In the last two, each piece of a unit writes its partial O / l and LSE to a
// slot of R rows; a second kernel merges each unit's slots.
struct DecodeProblem {
  int B, Sq, Scache, H, Hkv, D;
  int G, Pq, R, n_ptiles;  // tile geometry
  int causal, window;      // mask, evaluated at the query's position
  float scale, scale_log2;
  const int* lens;         // [B] keys per batch (clamped to [0, Scache]) or nullptr: Scache
  int splits, tiles_per_split;
  int persistent;
  int stream_k_min;
  float* lse;              // [B, H, Sq] fp32 or nullptr
  float* o_part;           // [slots, R, D] fp32 partial O / l (split modes)
  float* lse_part;         // [slots, R] fp32 partial LSE (split modes)
  unsigned* status;
  unsigned long long wait_limit_ns;
  int stall_probe;
  BshdStrides sq, sk, sv, so;  // layouts of q, the caches and out (zero: dense)
};

// Items (unit, KV-tile range, slot) one CTA of the KV-cache kernel can hold
// in its list; the plan keeps every CTA's share within it.
constexpr int kDecodeMaxItems = 80;

// Launches the KV-cache kernel (and, with splits > 1, the combine kernel).
cudaError_t launch_decode_bf16_tc(const DecodeProblem& p, void* out, const void* q, const void* k,
                                  const void* v, cudaStream_t stream);

// Tensor-core (tcgen05) bf16 forward. q/k/v/out are device pointers to
// 16-byte-aligned dense BSHD / BShD bf16 tensors. Returns a cudaError_t.
cudaError_t launch_fwd_bf16_tc(const FwdProblem& p, void* out, const void* q, const void* k,
                               const void* v, cudaStream_t stream);
// Query blocks (CTAs per (batch, head)) of that kernel for S queries and
// head dim D.
int fwd_bf16_tc_ctas(int S, int D);

// CUDA-core fp32 forward for fp32 tensors.
cudaError_t launch_fwd_f32_simt(const FwdProblem& p, float* out, const float* q, const float* k,
                                const float* v, cudaStream_t stream);

// fp32 forward on the tensor cores: every operand split into three bf16
// parts, six part products per contraction. q/out dense or strided BSHD
// (sq/so, zero: dense); k/v dense [B, S, Hkv, D], split into bf16 planes in
// a workspace of f32x3_workspace_bytes() bytes.
struct F32x3Problem {
  int B, S, H, Hkv, D;
  int causal, window;
  float scale, scale_log2;
  const float* q;
  const float* k;
  const float* v;
  float* out;
  float* lse;            // [B, H, S] or nullptr
  uint16_t* kp[3];       // K's bf16 planes (set by the launcher from the workspace)
  uint16_t* vp[3];       // V's bf16 planes
  BshdStrides sq, so;
  unsigned* status;
  unsigned long long wait_limit_ns;
  int stall_probe;
};
unsigned long long f32x3_workspace_bytes(int B, int S, int Hkv, int D);
cudaError_t launch_fwd_f32x3_tc(F32x3Problem p, void* workspace, cudaStream_t stream);

// Exact top-K per row (values descending in IEEE total order, ties by
// ascending index): chunk kernel (grid n_chunks x B) writing each chunk's top
// K keys to `cand` [B, n_chunks, K], then a merge kernel per row.
constexpr int kMaxTopK = 1024;
constexpr int kMaxTopkCandidates = 16384;  // n_chunks * K, the merge's shared memory
struct TopkProblem {
  const float* scores;   // [B, V] fp32, row_stride elements apart
  long long row_stride;
  int B, V, K;
  int chunk, n_chunks;   // elements per chunk (multiple of 1024), chunks per row
  uint64_t* cand;        // workspace: B * n_chunks * K keys
  float* values;         // [B, K]
  int* indices;          // [B, K]
};
cudaError_t launch_topk(const TopkProblem& p, cudaStream_t stream);

// Stores `msg` as the calling thread's fa_last_error_message().
void record_error_message(const char* msg);

// The bounded-wait limit every launch uses (fa_set_wait_timeout_ns).
unsigned long long wait_limit_ns();

// Raises `func`'s dynamic shared-memory limit to `bytes` once per device:
// `done` (one per kernel, zero-initialised static) keeps a bit per device
// index that has been set up. Later calls on that device cost one
// cudaGetDevice.
cudaError_t ensure_smem_attr(unsigned long long* done, const void* func, int bytes);

// Encodes a 4-D BSHD tensor map (dims D, heads, S, B; element strides `st`,
// D contiguous) for bf16 data with a {box_cols, box_heads, box_rows, 1} box:
// 64 columns with the 128-byte swizzle, or 32 with the 64-byte swizzle. Returns false on failure. Maps are cached, keyed on every
// argument (address, sizes, strides, box): a repeated call copies the cached
// map instead of encoding it again; fa_shutdown() empties the cache. With
// use_cache false the map is encoded and the cache neither read nor grown
// (no host allocation).
bool encode_bshd_tensor_map(CUtensorMap* map, const void* base, int B, int S, int heads, int D,
                            BshdStrides st, int box_heads = 1, int box_rows = 128,
                            bool use_cache = true, int box_cols = 64);

}  // namespace fa
