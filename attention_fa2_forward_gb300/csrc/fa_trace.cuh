// fa_trace.cuh -- compile-time event trace and bounds guards of the debug
// build (FA_TRACE=1, library libfa_mha_debug.so).
//
// Trace: each CTA of the prefill kernel owns kRoles x kEventsPerRole records
// of 16 bytes in a caller-provided device buffer; lane 0 of each warp (TMA
// producer, MMA issuer, the eight softmax warps) appends its events in
// program order:
//   x, y : %globaltimer (ns), low and high word -- comparable across SMs;
//   z    : low word of %clock64 of the SM -- cycle-accurate within a CTA;
//   w    : event code << 24 | 24-bit argument.
// A role that runs out of records drops the rest; records never written keep
// whatever the caller put there (zero it first). CTAs whose index lies past
// the buffer record nothing.
//
// Bounds guards: before an access whose index is computed at run time (a
// shared-memory ring slot, a tensor-memory column, an LSE element, a TMA
// store's first row) the debug build checks it against its extent; a failed
// check sets kStatusBoundsGuard in the status word and skips the access
// instead of trapping, so the context stays usable and the host reads the
// bit with fa_device_status / fa_stream_status.
//
// In the default build (FA_TRACE undefined or 0) every hook compiles to
// nothing and every guard to `true`.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

#ifndef FA_TRACE
#define FA_TRACE 0
#endif

namespace fa {
namespace trace {

// producer, MMA issuer, softmax warp 0 (tile 0) and 4 (tile 1), then softmax
// warps 1, 2, 3, 5, 6, 7
constexpr int kRoles = 10;
constexpr int kEventsPerRole = 256;
constexpr int kRecordBytes = 16;
constexpr unsigned long long kBytesPerCta =
    static_cast<unsigned long long>(kRoles) * kEventsPerRole * kRecordBytes;

enum Role : int { kRoleProducer = 0, kRoleMma = 1, kRoleSoftmax0 = 2, kRoleSoftmax1 = 3 };

// Role of softmax warp w (0-7) of the prefill kernel.
__host__ __device__ constexpr int softmax_role(int w) {
  return w == 0 ? kRoleSoftmax0 : w == 4 ? kRoleSoftmax1 : (w < 4 ? 3 + w : 2 + w);
}

// Event codes (the argument's meaning in brackets).
enum Code : uint32_t {
  kCtaStart = 1,      // producer role, first record [SM id]
  kQLoadIssued = 2,   // producer [Q tile]
  kKLoadIssued = 3,   // producer [KV tile j]
  kVLoadIssued = 4,   // producer [KV tile j]
  kQReady = 5,        // MMA issuer: every Q tile has landed [0]
  kSIssued = 6,       // MMA issuer [Q tile << 16 | KV tile j]
  kPvIssued = 7,      // MMA issuer [Q tile << 16 | KV tile j]
  kMmaDrained = 8,    // MMA issuer: every MMA has completed [0]
  kSReady = 9,        // softmax: S(j) is in tensor memory [KV tile j]
  kPReady = 10,       // softmax: P(j) stored, O corrected [KV tile j | rescaled << 23]
  kEpilogueStart = 11,  // softmax: O(final) is ready [0]
  kEpilogueEnd = 12,    // softmax: O stored, LSE written [0]
  kSLoaded = 13,        // softmax: S(j) is in registers [KV tile j]
  kMaxDone = 14,        // softmax: row maximum known [KV tile j]
  kExpDone = 15,        // softmax: P(j) computed, not yet stored [KV tile j]
  kPSeen = 16,          // MMA issuer: all of P(j) is in tensor memory [Q tile << 16 | j]
};

// Appends events of one role of one CTA. Construct in the thread that
// records; the other threads pass active = false.
struct Recorder {
#if FA_TRACE
  uint4* slot = nullptr;
  int n = 0;
  __device__ __forceinline__ Recorder(void* buf, long long ctas, int role, bool active) {
    if (active && buf != nullptr && static_cast<long long>(blockIdx.x) < ctas)
      slot = reinterpret_cast<uint4*>(buf) +
             (static_cast<long long>(blockIdx.x) * kRoles + role) * kEventsPerRole;
  }
  __device__ __forceinline__ void operator()(uint32_t code, uint32_t arg) {
    if (slot == nullptr || n >= kEventsPerRole) return;
    const uint64_t t = ptx::global_timer_ns();
    uint32_t clk;
    asm volatile("mov.u32 %0, %%clock;" : "=r"(clk));
    slot[n++] = make_uint4(static_cast<uint32_t>(t), static_cast<uint32_t>(t >> 32), clk,
                           (code << 24) | (arg & 0xffffffu));
  }
#else
  __device__ __forceinline__ Recorder(void*, long long, int, bool) {}
  __device__ __forceinline__ void operator()(uint32_t, uint32_t) {}
#endif
};

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t id;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
  return id;
}

// Bounds guard: `ok` in the default build is assumed; in the debug build a
// false `ok` records `bit` in the status word and returns false so that the
// caller skips the access.
__device__ __forceinline__ bool guard(bool ok, unsigned* status, unsigned bit) {
#if FA_TRACE
  if (!ok) {
    atomicOr(status, bit);
    return false;
  }
  return true;
#else
  (void)ok;
  (void)status;
  (void)bit;
  return true;
#endif
}

}  // namespace trace
}  // namespace fa
