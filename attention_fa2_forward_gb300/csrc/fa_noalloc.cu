// fa_noalloc.cu -- an entry point of the attention forward that allocates no
// device memory, for callers that cannot call cudaMalloc: code running where
// the allocator is owned by someone else (a framework's caching allocator, a
// memory pool sized up front), code that must not allocate on a latency-
// critical path, or code whose every allocation must be accounted for
// before it starts.
//
// The bf16 tensor-core kernel needs one piece of global memory besides its
// inputs and outputs: a status word in which a CTA records that it gave up
// on a bounded wait. fa_mha_no_cache allocates that word with cudaMalloc on
// its first call on a device. Here it lives instead in the file-scope array
// below, which every GPU that loads this library holds until the process
// exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "fa_mha.h"
#include "fa_internal.h"

namespace {

// Scratch of the allocation-free entry point. The kernel uses its first
// 4 bytes (the status word); the size is the stated maximum.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device

// Records the reason (read back with fa_last_error_message) and returns st.
fa_status_t noalloc_fail(fa_status_t st, const char* fmt, ...)
    __attribute__((format(printf, 2, 3)));
fa_status_t noalloc_fail(fa_status_t st, const char* fmt, ...) {
  char msg[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof(msg), fmt, ap);
  va_end(ap);
  fa::record_error_message(msg);
  return st;
}

// Scratch bytes the kernel needs for a problem: one status word, whatever the
// sizes are.
size_t scratch_bytes_needed(int /*B*/, int /*S*/, int /*H*/, int /*D*/) { return sizeof(unsigned); }

// Set-up, once per device, with that device current: resolve the device
// address of the scratch array. In host code `g_noalloc_scratch` is only a
// host-side stand-in for the symbol, never a device address.
fa_status_t scratch_address(int dev, unsigned** out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (err != cudaSuccess || ptr == nullptr)
      return noalloc_fail(FA_ERR_CUDA, "cudaGetSymbolAddress(scratch) on device %d: %s", dev,
                          cudaGetErrorString(err));
    g_scratch_addr[dev] = ptr;
  }
  *out = static_cast<unsigned*>(g_scratch_addr[dev]);
  return FA_OK;
}

}  // namespace

extern "C" fa_status_t fa_mha_no_cache_noalloc(void* out, float* lse, const void* q,
                                               const void* k, const void* v, int B, int S, int H,
                                               int Hkv, int D, float scale, int mask_kind,
                                               int local_window_size, void* stream,
                                               int check_status) {
  if (out == nullptr || q == nullptr || k == nullptr || v == nullptr)
    return noalloc_fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (B < 1 || S < 1 || H < 1 || Hkv < 1 || H % Hkv != 0)
    return noalloc_fail(FA_ERR_INVALID_ARG, "bad sizes B=%d S=%d H=%d Hkv=%d", B, S, H, Hkv);
  if (mask_kind != FA_MASK_NONE && mask_kind != FA_MASK_CAUSAL)
    return noalloc_fail(FA_ERR_INVALID_ARG, "unknown mask kind %d", mask_kind);
  if (local_window_size == 0 || local_window_size < -1)
    return noalloc_fail(FA_ERR_INVALID_ARG, "bad local_window_size %d", local_window_size);
  if (!std::isfinite(scale)) return noalloc_fail(FA_ERR_INVALID_ARG, "scale must be finite");
  if (scale < 0.f) return noalloc_fail(FA_ERR_UNSUPPORTED, "negative scale");
  if (D < 8 || D > 128 || D % 8 != 0)
    return noalloc_fail(FA_ERR_UNSUPPORTED, "head dim D=%d (multiples of 8 up to 128)", D);
  const long long elems_q = static_cast<long long>(B) * S * H * D;
  if (elems_q >= (1ll << 40) || static_cast<long long>(S) * H * D * 2 >= (1ll << 39) ||
      static_cast<long long>(B) * H * ((S + 255) / 256) > 0x7fffffffll)
    return noalloc_fail(FA_ERR_UNSUPPORTED, "problem too large");
  const size_t need = scratch_bytes_needed(B, S, H, D);
  if (need > kNoAllocScratchBytes)
    return noalloc_fail(FA_ERR_UNSUPPORTED,
                        "needs %zu scratch bytes; the allocation-free entry point has %zu", need,
                        kNoAllocScratchBytes);
  for (const void* p : {static_cast<const void*>(out), q, k, v})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
      return noalloc_fail(FA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned");
  if (lse != nullptr && reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return noalloc_fail(FA_ERR_UNSUPPORTED, "lse must be 4-byte aligned");

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return noalloc_fail(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(FA_ERR_UNSUPPORTED, "device %d", dev);
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return noalloc_fail(FA_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", major, minor);
  unsigned* status = nullptr;
  fa_status_t st = scratch_address(dev, &status);
  if (st != FA_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word must start
  // at zero for this call.
  err = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
  if (err != cudaSuccess)
    return noalloc_fail(FA_ERR_CUDA, "clearing the scratch status word: %s", cudaGetErrorString(err));

  fa::FwdProblem p;
  p.B = B;
  p.S = S;
  p.H = H;
  p.Hkv = Hkv;
  p.D = D;
  p.causal = mask_kind == FA_MASK_CAUSAL ? 1 : 0;
  p.window = local_window_size > 0 && local_window_size < S ? local_window_size : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lse = lse;
  p.status = status;
  p.wait_limit_ns = fa::wait_limit_ns();  // the limit fa_set_wait_timeout_ns sets
  p.stall_probe = 0;
  p.cache_maps = false;  // the tensor-map cache grows a host hash table
  // SM count for the persistent schedules (a device attribute: no allocation)
  cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, dev);
  err = fa::launch_fwd_bf16_tc(p, out, q, k, v, s);
  if (err != cudaSuccess)
    return noalloc_fail(FA_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(err));

  if (check_status) {
    unsigned word = 0;
    err = cudaMemcpyAsync(&word, status, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    if (err != cudaSuccess)
      return noalloc_fail(FA_ERR_CUDA, "reading the scratch status word: %s",
                          cudaGetErrorString(err));
    if (word & fa::kStatusWaitTimeout)
      return noalloc_fail(FA_ERR_TIMEOUT, "a CTA gave up on a bounded wait");
  }
  return FA_OK;
}
