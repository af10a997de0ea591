// fa_api.cu -- the C ABI declared in include/fa_mha.h: argument validation,
// per-device state (per-stream status words, cached tensor maps and kernel
// attributes), TMA tensor-map encoding and dispatch to the bf16 tensor-core
// kernel or the fp32 kernels, and the KV-cache and top-K entry points (work
// plans: tile geometry, key-range splits, chunks, workspace).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "fa_mha.h"
#include "fa_internal.h"
#include "fa_trace.cuh"
#include "topk_plan.h"

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;

std::mutex g_mutex;

// Status words, one per stream, per device: a device array of kStatusSlots
// words allocated on the device's first launch. Streams get slots in the
// order they are first used; once the array is full, further streams share
// its last word.
constexpr int kStatusSlots = 1024;
struct StatusPool {
  unsigned* words = nullptr;  // device, kStatusSlots words
  std::unordered_map<const void*, int> slot_of;
};
StatusPool g_pool[kMaxDevices];
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_stall_probe{0};
thread_local char t_message[512] = "";
// Debug build only: event trace buffer of the prefill kernel and the LSE
// bound its guard enforces (0: the LSE tensor's size).
std::atomic<void*> g_trace_buf{nullptr};
std::atomic<unsigned long long> g_trace_bytes{0};
std::atomic<long long> g_lse_limit{0};

fa_status_t fail(fa_status_t st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
fa_status_t fail(fa_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_message, sizeof(t_message), fmt, ap);
  va_end(ap);
  return st;
}

fa_status_t cuda_fail(cudaError_t err, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// bf16 runs any D that is a multiple of 8 (16-byte rows for TMA) up to 128 on
// the 64- or 128-column tensor-core kernels; fp32 has warp kernels for D/32
// columns per lane.
bool head_dim_supported(int D, int dtype) {
  if (dtype == FA_DTYPE_BF16) return D >= 8 && D <= 256 && D % 8 == 0;
  return D == 32 || D == 64 || D == 96 || D == 128;
}

// Columns the tensor-core kernels work on for a head dim D.
int padded_head_dim(int D) { return D <= 64 ? 64 : (D <= 128 ? 128 : 256); }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// Status word of `stream` on device `dev` (the current device), created on
// first use.
fa_status_t stream_status_word(int dev, const void* stream, unsigned** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  StatusPool& pool = g_pool[dev];
  if (pool.words == nullptr) {
    unsigned* p = nullptr;
    cudaError_t err = cudaMalloc(&p, kStatusSlots * sizeof(unsigned));
    if (err != cudaSuccess) return cuda_fail(err, "cudaMalloc(status words)");
    err = cudaMemset(p, 0, kStatusSlots * sizeof(unsigned));
    if (err == cudaSuccess) err = cudaDeviceSynchronize();
    if (err != cudaSuccess) {
      cudaFree(p);
      return cuda_fail(err, "cudaMemset(status words)");
    }
    pool.words = p;
  }
  auto it = pool.slot_of.find(stream);
  int slot;
  if (it != pool.slot_of.end()) {
    slot = it->second;
  } else {
    slot = static_cast<int>(pool.slot_of.size());
    if (slot >= kStatusSlots - 1) {
      slot = kStatusSlots - 1;  // shared by every stream past the first 1023
    } else {
      pool.slot_of.emplace(stream, slot);
    }
  }
  *out = pool.words + slot;
  return FA_OK;
}

// Status code for the bits of a status word.
fa_status_t status_from_bits(unsigned bits, const char* where) {
  if (bits & fa::kStatusWaitTimeout)
    return fail(FA_ERR_TIMEOUT, "a kernel on %s gave up on a bounded wait", where);
  if (bits & fa::kStatusBoundsGuard)
    return fail(FA_ERR_BOUNDS, "a bounds guard of the debug build skipped an access on %s", where);
  return FA_OK;
}

// Whether device `dev` is sm_103 (asked once per device).
fa_status_t check_arch(int dev) {
  static std::atomic<int> known[kMaxDevices];  // 0 unknown, 1 sm_103, 2 other
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device index %d", dev);
  int k = known[dev].load(std::memory_order_acquire);
  if (k == 1) return FA_OK;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) {
    known[dev].store(2, std::memory_order_release);
    return fail(FA_ERR_UNSUPPORTED, "built for sm_103a; device %d is sm_%d%d", dev, major, minor);
  }
  known[dev].store(1, std::memory_order_release);
  return FA_OK;
}

// Cache of encoded tensor maps, keyed on every encoding argument.
struct MapKey {
  const void* base;
  long long dims[4];
  long long strides[3];
  int box_heads, box_rows, box_cols, pad;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    // FNV-1a over the key's bytes (the key has no padding: checked below).
    const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ b[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
static_assert(sizeof(MapKey) == 8 + 4 * 8 + 3 * 8 + 4 * 4, "MapKey must have no padding");
constexpr size_t kMapCacheMax = 4096;  // entries; the cache is emptied when it would grow past
std::mutex g_map_mutex;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;

}  // namespace

namespace fa {

void record_error_message(const char* msg) { snprintf(t_message, sizeof(t_message), "%s", msg); }

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(); }

cudaError_t ensure_smem_attr(unsigned long long* done, const void* func, int bytes) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const bool cacheable = dev >= 0 && dev < 64;
  const unsigned long long bit = cacheable ? 1ull << dev : 0ull;
  if (cacheable && (__atomic_load_n(done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess && cacheable) __atomic_fetch_or(done, bit, __ATOMIC_RELEASE);
  return err;
}

bool encode_bshd_tensor_map(CUtensorMap* map, const void* base, int B, int S, int heads, int D,
                            BshdStrides st, int box_heads, int box_rows, bool use_cache,
                            int box_cols) {
  if (box_cols != 64 && box_cols != 32) return false;
  st = resolve_strides(st, S, heads, D);
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.base = base;
  key.dims[0] = D;
  key.dims[1] = heads;
  key.dims[2] = S;
  key.dims[3] = B;
  key.strides[0] = st.h;
  key.strides[1] = st.s;
  key.strides[2] = st.b;
  key.box_heads = box_heads;
  key.box_rows = box_rows;
  key.box_cols = box_cols;
  if (use_cache) {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
      *map = it->second;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.h) * 2,
                                 static_cast<cuuint64_t>(st.s) * 2,
                                 static_cast<cuuint64_t>(st.b) * 2};
  if (box_heads < 1 || box_heads > 256 || box_rows < 1 || box_rows > 256) return false;
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols),
                             static_cast<cuuint32_t>(box_heads),
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (!use_cache) return true;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
  g_map_cache.emplace(key, *map);
  return true;
}

}  // namespace fa

namespace {

// Validates the arguments, then launches the kernel of `dtype` on `stream`.
// `strides` (may be null: dense) holds the element strides along B, S, H of
// q, k, v and out, in that order.
// Argument checks of the no-cache forward (no CUDA call).
fa_status_t check_forward_args(void* out, float* lse, const void* q, const void* k, const void* v,
                               int B, int S, int H, int Hkv, int D, float scale, int mask_kind,
                               int local_window_size, int dtype,
                               const fa::BshdStrides* strides) {
  if (out == nullptr || q == nullptr || k == nullptr || v == nullptr)
    return fail(FA_ERR_INVALID_ARG, "null tensor pointer (out=%p q=%p k=%p v=%p)", out, q, k, v);
  if (B < 1 || S < 1 || H < 1 || Hkv < 1)
    return fail(FA_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d S=%d H=%d Hkv=%d)", B, S, H, Hkv);
  if (H % Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "H=%d is not a multiple of Hkv=%d", H, Hkv);
  if (mask_kind != FA_MASK_NONE && mask_kind != FA_MASK_CAUSAL)
    return fail(FA_ERR_INVALID_ARG, "unknown mask kind %d", mask_kind);
  if (local_window_size == 0 || local_window_size < -1)
    return fail(FA_ERR_INVALID_ARG, "local_window_size must be -1 or >= 1 (got %d)",
                local_window_size);
  if (!std::isfinite(scale))
    return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  if (scale < 0.f)
    return fail(FA_ERR_UNSUPPORTED, "negative scale is not supported");
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F32)
    return fail(FA_ERR_UNSUPPORTED, "dtype %d", dtype);
  if (!head_dim_supported(D, dtype))
    return fail(FA_ERR_UNSUPPORTED, "head dim D=%d (bf16: multiples of 8 up to 256; fp32: 32, 64, "
                "96, 128)", D);
  if (dtype == FA_DTYPE_BF16 && D > 128 && H / Hkv > 128)
    return fail(FA_ERR_UNSUPPORTED, "D > 128 needs H / Hkv <= 128 (got %d)", H / Hkv);
  const long long elems_q = static_cast<long long>(B) * S * H * D;
  const long long row_bytes = static_cast<long long>(S) * H * D * 2;
  if (elems_q >= (1ll << 40) || row_bytes >= (1ll << 39) ||
      static_cast<long long>(B) * H * ((S + 255) / 256) > 0x7fffffffll)
    return fail(FA_ERR_UNSUPPORTED, "problem too large (B=%d S=%d H=%d D=%d)", B, S, H, D);
  const uintptr_t need = dtype == FA_DTYPE_BF16 ? 16 : 4;
  if (!aligned(out, need) || !aligned(q, need) || !aligned(k, need) || !aligned(v, need) ||
      (lse != nullptr && !aligned(lse, 4)))
    return fail(FA_ERR_UNSUPPORTED, "tensors must be %u-byte aligned",
                static_cast<unsigned>(need));
  if (strides != nullptr) {
    static const char* const names[4] = {"q", "k", "v", "out"};
    for (int t = 0; t < 4; ++t) {
      const fa::BshdStrides& st = strides[t];
      if (st.b < 1 || st.s < 1 || st.h < 1)
        return fail(FA_ERR_INVALID_ARG, "%s strides must be >= 1 (got %lld, %lld, %lld)",
                    names[t], st.b, st.s, st.h);
      if (st.b >= (1ll << 38) || st.s >= (1ll << 38) || st.h >= (1ll << 38))
        return fail(FA_ERR_UNSUPPORTED, "%s strides too large", names[t]);
      if (dtype == FA_DTYPE_BF16 && (st.b % 8 || st.s % 8 || st.h % 8))
        return fail(FA_ERR_UNSUPPORTED,
                    "bf16 %s strides must be multiples of 8 elements (16 bytes) for TMA",
                    names[t]);
    }
  }
  return FA_OK;
}

fa_status_t current_sm_count(int* out);

fa_status_t forward(void* out, float* lse, const void* q, const void* k, const void* v, int B,
                    int S, int H, int Hkv, int D, float scale, int mask_kind,
                    int local_window_size, int dtype, void* stream,
                    const fa::BshdStrides* strides) {
  // ---- arguments (no CUDA call before these pass)
  fa_status_t st = check_forward_args(out, lse, q, k, v, B, S, H, Hkv, D, scale, mask_kind,
                                      local_window_size, dtype, strides);
  if (st != FA_OK) return st;

  // ---- device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if ((st = check_arch(dev)) != FA_OK) return st;
  unsigned* status = nullptr;
  if ((st = stream_status_word(dev, stream, &status)) != FA_OK) return st;

  fa::FwdProblem p;
  p.B = B;
  p.S = S;
  p.H = H;
  p.Hkv = Hkv;
  p.D = D;
  p.causal = mask_kind == FA_MASK_CAUSAL ? 1 : 0;
  // A window of S keys or more hides nothing.
  p.window = local_window_size > 0 && local_window_size < S ? local_window_size : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lse = lse;
  p.status = status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.stall_probe = g_stall_probe.load();
  if ((st = current_sm_count(&p.num_sms)) != FA_OK) return st;
  if (FA_TRACE) {
    p.trace = g_trace_buf.load();
    p.trace_ctas = p.trace != nullptr
                       ? static_cast<long long>(g_trace_bytes.load() / fa::trace::kBytesPerCta)
                       : 0;
    p.lse_limit = g_lse_limit.load();
  }
  if (strides != nullptr) {
    p.sq = strides[0];
    p.sk = strides[1];
    p.sv = strides[2];
    p.so = strides[3];
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == FA_DTYPE_BF16 && D > 128) {
    // Head dims above 128 run on the one-Q-tile kernel of the KV-cache path
    // (S double-buffered in tensor-memory columns 0-255, O in 256-511) with
    // every key present: Sq = S_cache = S, one split.
    fa::DecodeProblem dp{};
    dp.B = B;
    dp.Sq = S;
    dp.Scache = S;
    dp.H = H;
    dp.Hkv = Hkv;
    dp.D = D;
    dp.G = H / Hkv;
    dp.Pq = S < 128 / dp.G ? S : 128 / dp.G;
    dp.R = dp.G * dp.Pq;
    dp.n_ptiles = (S + dp.Pq - 1) / dp.Pq;
    dp.causal = p.causal;
    dp.window = p.window;
    dp.scale = p.scale;
    dp.scale_log2 = p.scale_log2;
    dp.lens = nullptr;
    dp.splits = 1;
    dp.tiles_per_split = (S + 127) / 128;
    dp.lse = lse;
    dp.status = status;
    dp.wait_limit_ns = p.wait_limit_ns;
    dp.stall_probe = p.stall_probe;
    dp.sq = p.sq;
    dp.sk = p.sk;
    dp.sv = p.sv;
    dp.so = p.so;
    if (static_cast<long long>(Hkv) * dp.n_ptiles * B > 0x7fffffffll)
      return fail(FA_ERR_UNSUPPORTED, "problem too large (grid)");
    err = fa::launch_decode_bf16_tc(dp, out, q, k, v, s);
    if (err != cudaSuccess) return cuda_fail(err, "bf16 tensor-core kernel launch (D > 128)");
  } else if (dtype == FA_DTYPE_BF16) {
    err = fa::launch_fwd_bf16_tc(p, out, q, k, v, s);
    if (err != cudaSuccess) return cuda_fail(err, "bf16 tensor-core kernel launch");
  } else {
    err = fa::launch_fwd_f32_simt(p, static_cast<float*>(out), static_cast<const float*>(q),
                                  static_cast<const float*>(k), static_cast<const float*>(v), s);
    if (err != cudaSuccess) return cuda_fail(err, "fp32 kernel launch");
  }
  return FA_OK;
}

// ------------------------------------------------------------- KV cache

// How the KV-cache kernel cuts the work (see fa_mha_kv_cache_plan).
struct KvPlan {
  int G, Pq, R, n_ptiles;
  int window;  // effective window (0: none)
  int splits, tiles_per_split;
  int ctas;          // persistent CTAs (0: a CTA per unit)
  int stream_k_min;  // > 0: stream-K sharing, quotas of at least this many tiles
  unsigned long long o_part_bytes, workspace_bytes;
};

constexpr int kMaxSplits = 128;
// Stream-K sharing: persistent CTAs per SM count (27/32: 128 of 152 SMs) --
// on a 152-SM GB300 the streaming CTAs' aggregate HBM throughput peaks at
// 128 CTAs and falls past it (one 131072-key cache, 8 KV heads: 6.1 TB/s at
// 128, 5.7 at 152) -- and the smallest quota in KV tiles.
constexpr long long kStreamKCtasNum = 27, kStreamKCtasDen = 32;
constexpr int kStreamKMinTiles = 2;

unsigned long long align256(unsigned long long x) { return (x + 255ull) & ~255ull; }

// Validates the size, mask and split arguments of the KV-cache entry points.
fa_status_t check_kv_args(int B, int Sq, int S_cache, int H, int Hkv, int D, int mask_kind,
                          int local_window_size, int num_splits) {
  if (B < 1 || Sq < 1 || S_cache < 1 || H < 1 || Hkv < 1)
    return fail(FA_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d Sq=%d S_cache=%d H=%d Hkv=%d)", B,
                Sq, S_cache, H, Hkv);
  if (H % Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "H=%d is not a multiple of Hkv=%d", H, Hkv);
  if (mask_kind != FA_MASK_NONE && mask_kind != FA_MASK_CAUSAL)
    return fail(FA_ERR_INVALID_ARG, "unknown mask kind %d", mask_kind);
  if (local_window_size == 0 || local_window_size < -1)
    return fail(FA_ERR_INVALID_ARG, "local_window_size must be -1 or >= 1 (got %d)",
                local_window_size);
  if (num_splits < 0) return fail(FA_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (!head_dim_supported(D, FA_DTYPE_BF16))
    return fail(FA_ERR_UNSUPPORTED, "head dim D=%d (multiples of 8 up to 256)", D);
  if (H / Hkv > 128)
    return fail(FA_ERR_UNSUPPORTED, "H / Hkv = %d query heads per KV head (at most 128)", H / Hkv);
  const long long q_elems = static_cast<long long>(B) * Sq * H * D;
  const long long c_elems = static_cast<long long>(B) * S_cache * Hkv * D;
  if (q_elems >= (1ll << 40) || c_elems >= (1ll << 40) ||
      static_cast<long long>(S_cache) * Hkv * D * 2 >= (1ll << 39))
    return fail(FA_ERR_UNSUPPORTED, "problem too large");
  return FA_OK;
}

KvPlan make_kv_plan(int B, int Sq, int S_cache, int H, int Hkv, int D, int causal,
                    int local_window_size, int num_splits, int num_sms) {
  KvPlan k{};
  k.G = H / Hkv;
  k.Pq = Sq < 128 / k.G ? Sq : 128 / k.G;
  k.R = k.G * k.Pq;
  k.n_ptiles = (Sq + k.Pq - 1) / k.Pq;
  // A window reaching past every key of the cache hides nothing.
  k.window = local_window_size > 0 && local_window_size < S_cache ? local_window_size : 0;
  // Most KV tiles one position tile can need.
  const long long all_tiles = (S_cache + 127) / 128;
  long long max_tiles = all_tiles;
  if (k.window > 0) {
    const long long span = causal ? (k.Pq - 1ll + k.window) : (k.Pq + 2ll * k.window - 2);
    max_tiles = (span + 127) / 128 + 1;
    if (max_tiles > all_tiles) max_tiles = all_tiles;
  }
  const long long units = static_cast<long long>(B) * Hkv * k.n_ptiles;
  const unsigned long long d_pad = padded_head_dim(D);  // the kernel's padded row
  unsigned long long slots = 0;                          // partial-result slots of R rows
  if (num_splits == 0) {
    // Auto. Units (batch x KV head x position tile) that fill half the SMs
    // stream best whole (one CTA each, no combine). Fewer are shared out
    // stream-K fashion: every persistent CTA takes an equal quota of all the
    // units' KV tiles (the lengths, and so the total, are known only on the
    // device); a unit is cut at the quota boundaries inside it.
    if (2 * units >= num_sms || max_tiles <= kStreamKMinTiles) {
      k.splits = 1;
      k.tiles_per_split = static_cast<int>(max_tiles);
    } else if (units / Hkv > fa::kDecodeMaxItems) {
      // More position-tile groups than a CTA's item list holds (a device with
      // many SMs): fixed splits, about two per SM.
      num_splits = static_cast<int>((2ll * num_sms + units - 1) / units);
      if (num_splits < 2) num_splits = 2;
    } else {
      // CTA groups of Hkv CTAs (one per KV head) share each quota.
      long long ctas = (kStreamKCtasNum * num_sms) / kStreamKCtasDen / Hkv * Hkv;
      if (ctas < Hkv) ctas = Hkv;
      k.ctas = static_cast<int>(ctas);
      k.stream_k_min = kStreamKMinTiles;
      k.tiles_per_split = static_cast<int>(max_tiles);
      // Pieces one unit may be cut into: one per CTA group at most, one per
      // tile.
      const long long groups_of_ctas = ctas / Hkv;
      k.splits = static_cast<int>(groups_of_ctas < max_tiles ? groups_of_ctas : max_tiles);
      if (k.splits < 2) k.splits = 2;
      // Pieces in all: one per unit with keys, plus one per unit of a group
      // that a quota boundary cuts.
      slots = static_cast<unsigned long long>(units + ctas);
    }
  }
  if (num_splits > 0) {
    // Fixed splits: the unit's tiles cut in `splits` even ranges; persistent
    // CTAs (one per SM at most) take every CTA-count-th range with keys.
    long long splits = num_splits;
    if (splits > kMaxSplits) splits = kMaxSplits;
    if (splits > max_tiles) splits = max_tiles;
    k.tiles_per_split = static_cast<int>((max_tiles + splits - 1) / splits);
    k.splits = static_cast<int>((max_tiles + k.tiles_per_split - 1) / k.tiles_per_split);
    if (k.splits > 1) {
      // One CTA per SM; more when a CTA's share would not fit its list.
      const long long ranges = units * k.splits;
      long long ctas = ranges < num_sms ? ranges : num_sms;
      const long long need = (ranges + fa::kDecodeMaxItems - 1) / fa::kDecodeMaxItems;
      if (ctas < need) ctas = need;
      k.ctas = static_cast<int>(ctas);
      slots = static_cast<unsigned long long>(ranges);
    }
  }
  if (slots > 0) {
    k.o_part_bytes = align256(slots * k.R * d_pad * 4ull);
    k.workspace_bytes = k.o_part_bytes + align256(slots * k.R * 4ull);
  }
  return k;
}

// SM count of the current device (asked once per device).
fa_status_t current_sm_count(int* out) {
  static std::atomic<int> known[kMaxDevices];  // 0: not asked yet
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev >= 0 && dev < kMaxDevices && (*out = known[dev].load(std::memory_order_acquire)) > 0)
    return FA_OK;
  err = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaDeviceGetAttribute(SM count)");
  if (dev >= 0 && dev < kMaxDevices) known[dev].store(*out, std::memory_order_release);
  return FA_OK;
}

// ---------------------------------------------------------------- top-K

struct TopkPlan {
  int chunk, n_chunks;
  unsigned long long workspace_bytes;
};

// Chunks per row: about two CTAs per SM over the whole batch, chunks of a
// multiple of 2048 elements (8 warps x 256-element steps), and at most 4096
// candidates per row for the merge.
TopkPlan make_topk_plan(int B, int V, int K, int num_sms) {
  constexpr long long kStep = 2048;
  // At most one wave of chunk CTAs (two resident per SM): a second, partial
  // wave would take as long as a full one.
  long long chunks = 2ll * num_sms / B;
  const long long by_merge = 4096 / K > 0 ? 4096 / K : 1;
  if (chunks > by_merge) chunks = by_merge;
  if (chunks < 1) chunks = 1;
  long long chunk = (V + chunks - 1) / chunks;
  chunk = (chunk + kStep - 1) / kStep * kStep;
  TopkPlan t;
  t.chunk = static_cast<int>(chunk);
  t.n_chunks = static_cast<int>((V + chunk - 1) / chunk);
  // A row of one chunk is finished by its chunk CTA, a row of 2, 4 or 8 (K up
  // to 128) by its cluster's first CTA: no candidates to keep in either case.
  t.workspace_bytes = fa::topk_clustered(t.n_chunks, K)
                          ? 0ull
                          : static_cast<unsigned long long>(B) * t.n_chunks * K * 8ull;
  return t;
}

fa_status_t check_topk_args(int B, int V, int K) {
  if (B < 1 || V < 1) return fail(FA_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d V=%d)", B, V);
  if (K < 1 || K > V) return fail(FA_ERR_INVALID_ARG, "K must be in [1, V] (K=%d V=%d)", K, V);
  if (K > fa::kMaxTopK) return fail(FA_ERR_UNSUPPORTED, "K=%d (at most %d)", K, fa::kMaxTopK);
  if (B > 65535) return fail(FA_ERR_UNSUPPORTED, "B=%d rows (at most 65535)", B);
  if (V > (1 << 30)) return fail(FA_ERR_UNSUPPORTED, "V=%d (at most 2^30)", V);
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status_t fa_topk_plan(int B, int V, int K, int num_sms, int* chunks_out,
                         unsigned long long* workspace_bytes_out) {
  if (chunks_out == nullptr || workspace_bytes_out == nullptr)
    return fail(FA_ERR_INVALID_ARG, "null output pointer");
  fa_status_t st = check_topk_args(B, V, K);
  if (st != FA_OK) return st;
  if (num_sms < 0) return fail(FA_ERR_INVALID_ARG, "num_sms must be >= 0");
  if (num_sms == 0 && (st = current_sm_count(&num_sms)) != FA_OK) return st;
  const TopkPlan t = make_topk_plan(B, V, K, num_sms);
  *chunks_out = t.n_chunks;
  *workspace_bytes_out = t.workspace_bytes;
  return FA_OK;
}

fa_status_t fa_topk(float* values, int* indices, const float* scores, int B, int V,
                    long long row_stride, int K, void* workspace,
                    unsigned long long workspace_bytes, void* stream) {
  if (values == nullptr || indices == nullptr || scores == nullptr)
    return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  fa_status_t st = check_topk_args(B, V, K);
  if (st != FA_OK) return st;
  if (row_stride < V) return fail(FA_ERR_INVALID_ARG, "row_stride %lld < V %d", row_stride, V);
  if (row_stride >= (1ll << 40)) return fail(FA_ERR_UNSUPPORTED, "row_stride too large");
  if (!aligned(values, 4) || !aligned(indices, 4) || !aligned(scores, 4) ||
      (workspace != nullptr && !aligned(workspace, 8)))
    return fail(FA_ERR_UNSUPPORTED, "buffers must be 4-byte aligned (workspace 8)");
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if ((st = check_arch(dev)) != FA_OK) return st;
  if ((st = current_sm_count(&sms)) != FA_OK) return st;
  const TopkPlan t = make_topk_plan(B, V, K, sms);
  if (t.workspace_bytes > 0 && (workspace == nullptr || workspace_bytes < t.workspace_bytes))
    return fail(FA_ERR_INVALID_ARG, "workspace of %llu bytes needed, %llu given",
                t.workspace_bytes, workspace != nullptr ? workspace_bytes : 0ull);
  fa::TopkProblem p;
  p.scores = scores;
  p.row_stride = row_stride;
  p.B = B;
  p.V = V;
  p.K = K;
  p.chunk = t.chunk;
  p.n_chunks = t.n_chunks;
  p.cand = static_cast<uint64_t*>(workspace);
  p.values = values;
  p.indices = indices;
  err = fa::launch_topk(p, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "top-K kernel launch");
  return FA_OK;
}

unsigned long long fa_mha_no_cache_f32_tc_workspace(int B, int S, int Hkv, int D) {
  if (B < 1 || S < 1 || Hkv < 1 || (D != 64 && D != 128)) return 0ull;
  return fa::f32x3_workspace_bytes(B, S, Hkv, D);
}

fa_status_t fa_mha_no_cache_f32_tc(float* out, float* lse, const float* q, const float* k,
                                   const float* v, int B, int S, int H, int Hkv, int D, float scale,
                                   int mask_kind, int local_window_size, void* workspace,
                                   unsigned long long workspace_bytes, void* stream) {
  if (out == nullptr || q == nullptr || k == nullptr || v == nullptr)
    return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (B < 1 || S < 1 || H < 1 || Hkv < 1)
    return fail(FA_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d S=%d H=%d Hkv=%d)", B, S, H, Hkv);
  if (H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H=%d is not a multiple of Hkv=%d", H, Hkv);
  if (mask_kind != FA_MASK_NONE && mask_kind != FA_MASK_CAUSAL)
    return fail(FA_ERR_INVALID_ARG, "unknown mask kind %d", mask_kind);
  if (local_window_size == 0 || local_window_size < -1)
    return fail(FA_ERR_INVALID_ARG, "local_window_size must be -1 or >= 1 (got %d)",
                local_window_size);
  if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  if (scale < 0.f) return fail(FA_ERR_UNSUPPORTED, "negative scale is not supported");
  if (D != 64 && D != 128) return fail(FA_ERR_UNSUPPORTED, "head dim D=%d (64 or 128)", D);
  const long long elems_q = static_cast<long long>(B) * S * H * D;
  if (elems_q >= (1ll << 40) || static_cast<long long>(S) * H * D * 4 >= (1ll << 39) ||
      static_cast<long long>(B) * H * ((S + 127) / 128) > 0x7fffffffll)
    return fail(FA_ERR_UNSUPPORTED, "problem too large");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      (lse != nullptr && !aligned(lse, 4)) || (workspace != nullptr && !aligned(workspace, 256)))
    return fail(FA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned (workspace 256)");
  const unsigned long long need = fa::f32x3_workspace_bytes(B, S, Hkv, D);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "workspace of %llu bytes needed, %llu given", need,
                workspace != nullptr ? workspace_bytes : 0ull);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  fa_status_t st = check_arch(dev);
  if (st != FA_OK) return st;
  unsigned* status = nullptr;
  if ((st = stream_status_word(dev, stream, &status)) != FA_OK) return st;
  fa::F32x3Problem p{};
  p.B = B;
  p.S = S;
  p.H = H;
  p.Hkv = Hkv;
  p.D = D;
  p.causal = mask_kind == FA_MASK_CAUSAL ? 1 : 0;
  p.window = local_window_size > 0 && local_window_size < S ? local_window_size : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.lse = lse;
  p.status = status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.stall_probe = g_stall_probe.load();
  err = fa::launch_fwd_f32x3_tc(p, workspace, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "fp32 tensor-core kernel launch");
  return FA_OK;
}

fa_status_t fa_mha_kv_cache_plan(int B, int Sq, int S_cache, int H, int Hkv, int D, int mask_kind,
                                 int local_window_size, int num_splits, int num_sms,
                                 int* splits_out, unsigned long long* workspace_bytes_out) {
  if (splits_out == nullptr || workspace_bytes_out == nullptr)
    return fail(FA_ERR_INVALID_ARG, "null output pointer");
  fa_status_t st = check_kv_args(B, Sq, S_cache, H, Hkv, D, mask_kind, local_window_size,
                                 num_splits);
  if (st != FA_OK) return st;
  if (num_sms < 0) return fail(FA_ERR_INVALID_ARG, "num_sms must be >= 0");
  if (num_sms == 0 && (st = current_sm_count(&num_sms)) != FA_OK) return st;
  const KvPlan k = make_kv_plan(B, Sq, S_cache, H, Hkv, D, mask_kind == FA_MASK_CAUSAL,
                                local_window_size, num_splits, num_sms);
  *splits_out = k.splits;
  *workspace_bytes_out = k.workspace_bytes;
  return FA_OK;
}

fa_status_t fa_mha_kv_cache(void* out, float* lse, const void* q, const void* k_cache,
                            const void* v_cache, const int* cache_lens, int B, int Sq,
                            int S_cache, int H, int Hkv, int D, float scale, int mask_kind,
                            int local_window_size, int num_splits, void* workspace,
                            unsigned long long workspace_bytes, int dtype, void* stream) {
  if (out == nullptr || q == nullptr || k_cache == nullptr || v_cache == nullptr)
    return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  fa_status_t st = check_kv_args(B, Sq, S_cache, H, Hkv, D, mask_kind, local_window_size,
                                 num_splits);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  if (scale < 0.f) return fail(FA_ERR_UNSUPPORTED, "negative scale is not supported");
  if (dtype != FA_DTYPE_BF16)
    return fail(FA_ERR_UNSUPPORTED, "the KV-cache entry point takes bf16 only (dtype %d)", dtype);
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      (lse != nullptr && !aligned(lse, 4)) || (cache_lens != nullptr && !aligned(cache_lens, 4)) ||
      (workspace != nullptr && !aligned(workspace, 16)))
    return fail(FA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned (lse, cache_lens: 4)");

  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if ((st = check_arch(dev)) != FA_OK) return st;
  if ((st = current_sm_count(&sms)) != FA_OK) return st;
  const KvPlan plan = make_kv_plan(B, Sq, S_cache, H, Hkv, D, mask_kind == FA_MASK_CAUSAL,
                                   local_window_size, num_splits, sms);
  if (plan.workspace_bytes > 0 && (workspace == nullptr || workspace_bytes < plan.workspace_bytes))
    return fail(FA_ERR_INVALID_ARG, "workspace of %llu bytes needed (%d splits), %llu given",
                plan.workspace_bytes, plan.splits, workspace != nullptr ? workspace_bytes : 0ull);
  // Units (a CTA each when unsplit) and partial slots must be indexable.
  if (static_cast<long long>(plan.splits) * Hkv * plan.n_ptiles * B > 0x7fffffffll)
    return fail(FA_ERR_UNSUPPORTED, "problem too large (grid)");
  unsigned* status = nullptr;
  if ((st = stream_status_word(dev, stream, &status)) != FA_OK) return st;

  fa::DecodeProblem p{};
  p.B = B;
  p.Sq = Sq;
  p.Scache = S_cache;
  p.H = H;
  p.Hkv = Hkv;
  p.D = D;
  p.G = plan.G;
  p.Pq = plan.Pq;
  p.R = plan.R;
  p.n_ptiles = plan.n_ptiles;
  p.causal = mask_kind == FA_MASK_CAUSAL ? 1 : 0;
  p.window = plan.window;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lens = cache_lens;
  p.splits = plan.splits;
  p.tiles_per_split = plan.tiles_per_split;
  p.persistent = plan.splits > 1 ? plan.ctas : 0;
  p.stream_k_min = plan.stream_k_min;
  p.lse = lse;
  if (plan.splits > 1) {
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.o_part_bytes);
  }
  p.status = status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.stall_probe = g_stall_probe.load();
  err = fa::launch_decode_bf16_tc(p, out, q, k_cache, v_cache, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "KV-cache kernel launch");
  return FA_OK;
}

fa_status_t fa_mha_no_cache(void* out, float* lse, const void* q, const void* k, const void* v,
                            int B, int S, int H, int Hkv, int D, float scale, int mask_kind,
                            int local_window_size, int dtype, void* stream) {
  return forward(out, lse, q, k, v, B, S, H, Hkv, D, scale, mask_kind, local_window_size, dtype,
                 stream, nullptr);
}

fa_status_t fa_mha_no_cache_strided(void* out, float* lse, const void* q, const void* k,
                                    const void* v, int B, int S, int H, int Hkv, int D,
                                    const long long* q_strides, const long long* k_strides,
                                    const long long* v_strides, const long long* out_strides,
                                    float scale, int mask_kind, int local_window_size, int dtype,
                                    void* stream) {
  if (q_strides == nullptr || k_strides == nullptr || v_strides == nullptr ||
      out_strides == nullptr)
    return fail(FA_ERR_INVALID_ARG, "null stride array");
  const long long* in[4] = {q_strides, k_strides, v_strides, out_strides};
  fa::BshdStrides st[4];
  for (int t = 0; t < 4; ++t) {
    st[t].b = in[t][0];
    st[t].s = in[t][1];
    st[t].h = in[t][2];
  }
  return forward(out, lse, q, k, v, B, S, H, Hkv, D, scale, mask_kind, local_window_size, dtype,
                 stream, st);
}

// Device workspace of fa_mha_no_cache_host: q, k, v, out, lse, then (fp32
// with D 64 or 128) the tensor-core path's bf16 planes, each 256-byte aligned.
struct HostLayout {
  unsigned long long q, k, v, out, lse, planes, total;
};
HostLayout host_layout(int B, int S, int H, int Hkv, int D, int dtype) {
  const unsigned long long e = dtype == FA_DTYPE_BF16 ? 2ull : 4ull;
  const unsigned long long q_bytes = static_cast<unsigned long long>(B) * S * H * D * e;
  const unsigned long long kv_bytes = static_cast<unsigned long long>(B) * S * Hkv * D * e;
  const unsigned long long lse_bytes = static_cast<unsigned long long>(B) * H * S * 4ull;
  HostLayout l{};
  l.q = 0;
  l.k = align256(l.q + q_bytes);
  l.v = align256(l.k + kv_bytes);
  l.out = align256(l.v + kv_bytes);
  l.lse = align256(l.out + q_bytes);
  l.planes = align256(l.lse + lse_bytes);
  const bool f32_tc = dtype == FA_DTYPE_F32 && (D == 64 || D == 128);
  l.total = l.planes + (f32_tc ? fa::f32x3_workspace_bytes(B, S, Hkv, D) : 0ull);
  return l;
}

unsigned long long fa_mha_no_cache_host_workspace(int B, int S, int H, int Hkv, int D,
                                                  int dtype) {
  if (B < 1 || S < 1 || H < 1 || Hkv < 1 || D < 1 ||
      (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F32))
    return 0ull;
  return host_layout(B, S, H, Hkv, D, dtype).total;
}

fa_status_t fa_mha_no_cache_host(void* out, float* lse, const void* q, const void* k,
                                 const void* v, int B, int S, int H, int Hkv, int D, float scale,
                                 int mask_kind, int local_window_size, int dtype, void* workspace,
                                 unsigned long long workspace_bytes, void* stream) {
  if (out == nullptr || q == nullptr || k == nullptr || v == nullptr)
    return fail(FA_ERR_INVALID_ARG, "null host pointer (out=%p q=%p k=%p v=%p)", out, q, k, v);
  if (workspace == nullptr || !aligned(workspace, 256))
    return fail(FA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device buffer");
  char* ws = static_cast<char*>(workspace);
  fa_status_t st = FA_OK;
  if (B >= 1 && S >= 1 && H >= 1 && Hkv >= 1 && D >= 1) {
    const HostLayout l = host_layout(B, S, H, Hkv, D, dtype);
    // The device-side arguments the launch will get (checked before any copy).
    st = check_forward_args(ws + l.out, lse != nullptr ? reinterpret_cast<float*>(ws + l.lse)
                                                       : nullptr,
                            ws + l.q, ws + l.k, ws + l.v, B, S, H, Hkv, D, scale, mask_kind,
                            local_window_size, dtype, nullptr);
    if (st == FA_OK && workspace_bytes < l.total)
      st = fail(FA_ERR_INVALID_ARG, "workspace of %llu bytes needed, %llu given", l.total,
                workspace_bytes);
  } else {
    st = check_forward_args(out, lse, q, k, v, B, S, H, Hkv, D, scale, mask_kind,
                            local_window_size, dtype, nullptr);
  }
  if (st != FA_OK) return st;
  const HostLayout l = host_layout(B, S, H, Hkv, D, dtype);
  const unsigned long long e = dtype == FA_DTYPE_BF16 ? 2ull : 4ull;
  const unsigned long long q_bytes = static_cast<unsigned long long>(B) * S * H * D * e;
  const unsigned long long kv_bytes = static_cast<unsigned long long>(B) * S * Hkv * D * e;
  const unsigned long long lse_bytes = static_cast<unsigned long long>(B) * H * S * 4ull;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  if ((err = cudaMemcpyAsync(ws + l.q, q, q_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (err = cudaMemcpyAsync(ws + l.k, k, kv_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (err = cudaMemcpyAsync(ws + l.v, v, kv_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(err, "cudaMemcpyAsync (inputs to the device)");
  float* lse_d = lse != nullptr ? reinterpret_cast<float*>(ws + l.lse) : nullptr;
  if (dtype == FA_DTYPE_F32 && (D == 64 || D == 128)) {
    st = fa_mha_no_cache_f32_tc(reinterpret_cast<float*>(ws + l.out), lse_d,
                                reinterpret_cast<const float*>(ws + l.q),
                                reinterpret_cast<const float*>(ws + l.k),
                                reinterpret_cast<const float*>(ws + l.v), B, S, H, Hkv, D, scale,
                                mask_kind, local_window_size, ws + l.planes,
                                l.total - l.planes, stream);
  } else {
    st = forward(ws + l.out, lse_d, ws + l.q, ws + l.k, ws + l.v, B, S, H, Hkv, D, scale,
                 mask_kind, local_window_size, dtype, stream, nullptr);
  }
  if (st != FA_OK) return st;
  if ((err = cudaMemcpyAsync(out, ws + l.out, q_bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(err, "cudaMemcpyAsync (output to the host)");
  if (lse != nullptr &&
      (err = cudaMemcpyAsync(lse, lse_d, lse_bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(err, "cudaMemcpyAsync (lse to the host)");
  return FA_OK;
}

fa_status_t fa_device_status(int device, int clear) {
  if (device < 0 || device >= kMaxDevices)
    return fail(FA_ERR_INVALID_ARG, "device index %d", device);
  int prev = 0;
  cudaError_t err = cudaGetDevice(&prev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (prev != device && (err = cudaSetDevice(device)) != cudaSuccess)
    return cuda_fail(err, "cudaSetDevice");
  fa_status_t result = FA_OK;
  err = cudaDeviceSynchronize();
  if (err != cudaSuccess) {
    result = cuda_fail(err, "cudaDeviceSynchronize");
  } else {
    // The lock keeps fa_shutdown from freeing the words while they are read.
    std::lock_guard<std::mutex> lock(g_mutex);
    unsigned* words = g_pool[device].words;
    if (words != nullptr) {
      static unsigned host[kStatusSlots];
      err = cudaMemcpy(host, words, sizeof(host), cudaMemcpyDeviceToHost);
      if (err != cudaSuccess) {
        result = cuda_fail(err, "cudaMemcpy(status words)");
      } else {
        unsigned bits = 0;
        for (int i = 0; i < kStatusSlots; ++i) bits |= host[i];
        if (clear && bits != 0 &&
            (err = cudaMemset(words, 0, kStatusSlots * sizeof(unsigned))) != cudaSuccess)
          result = cuda_fail(err, "cudaMemset(status words)");
        else if (clear && bits != 0 && (err = cudaDeviceSynchronize()) != cudaSuccess)
          result = cuda_fail(err, "cudaDeviceSynchronize");
        else
          result = status_from_bits(bits, "the device");
      }
    }
  }
  if (prev != device) cudaSetDevice(prev);
  return result;
}

fa_status_t fa_stream_status(void* stream, int clear) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device index %d", dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* word = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    StatusPool& pool = g_pool[dev];
    if (pool.words != nullptr) {
      auto it = pool.slot_of.find(stream);
      if (it != pool.slot_of.end())
        word = pool.words + it->second;
      else if (static_cast<int>(pool.slot_of.size()) >= kStatusSlots - 1)
        word = pool.words + (kStatusSlots - 1);
    }
  }
  unsigned bits = 0;
  if (word != nullptr) {
    err = cudaMemcpyAsync(&bits, word, sizeof(bits), cudaMemcpyDeviceToHost, s);
    if (err != cudaSuccess) return cuda_fail(err, "cudaMemcpyAsync(status word)");
    if (clear && (err = cudaMemsetAsync(word, 0, sizeof(unsigned), s)) != cudaSuccess)
      return cuda_fail(err, "cudaMemsetAsync(status word)");
  }
  err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return cuda_fail(err, "cudaStreamSynchronize");
  return status_from_bits(bits, "this stream");
}

fa_status_t fa_trace_set_buffer(void* buf, unsigned long long bytes) {
  if (!FA_TRACE) {
    if (buf == nullptr) return FA_OK;
    return fail(FA_ERR_UNSUPPORTED, "event traces need the debug build (libfa_mha_debug.so)");
  }
  if (buf != nullptr && (reinterpret_cast<uintptr_t>(buf) % 16 != 0))
    return fail(FA_ERR_INVALID_ARG, "trace buffer must be 16-byte aligned");
  g_trace_buf.store(nullptr);
  g_trace_bytes.store(buf != nullptr ? bytes : 0ull);
  g_trace_buf.store(buf);
  return FA_OK;
}

unsigned long long fa_trace_bytes_per_cta(void) { return FA_TRACE ? fa::trace::kBytesPerCta : 0ull; }

long long fa_trace_ctas(int B, int S, int H, int D) {
  if (B < 1 || S < 1 || H < 1 || D < 8 || D > 128) return 0;
  return static_cast<long long>(fa::fwd_bf16_tc_ctas(S, D)) * H * B;
}

fa_status_t fa_debug_set_lse_limit(long long elems) {
  if (!FA_TRACE) return fail(FA_ERR_UNSUPPORTED, "bounds guards need the debug build");
  if (elems < 0) return fail(FA_ERR_INVALID_ARG, "limit must be >= 0");
  g_lse_limit.store(elems);
  return FA_OK;
}

unsigned long long fa_set_wait_timeout_ns(unsigned long long ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? kDefaultWaitLimitNs : ns);
}

int fa_set_stall_probe(int enable) { return g_stall_probe.exchange(enable ? 1 : 0); }

const char* fa_status_string(fa_status_t status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS";
    default: return "FA_ERR_UNKNOWN";
  }
}

const char* fa_last_error_message(void) { return t_message; }

int fa_version(void) { return kVersion; }

void fa_shutdown(void) {
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    int prev = -1;
    cudaGetDevice(&prev);
    for (int d = 0; d < kMaxDevices; ++d) {
      StatusPool& pool = g_pool[d];
      if (pool.words != nullptr) {
        if (cudaSetDevice(d) == cudaSuccess) cudaFree(pool.words);
        pool.words = nullptr;
      }
      pool.slot_of.clear();
    }
    if (prev >= 0) cudaSetDevice(prev);
  }
  std::lock_guard<std::mutex> lock(g_map_mutex);
  g_map_cache.clear();
}

}  // extern "C"
