// fa_tile.cuh -- per-row arithmetic on the score columns of one 128-key tile,
// shared by the tensor-core kernels (prefill and KV-cache). A softmax thread
// owns N columns of one query row (one tensor-memory lane): all 128 in the
// KV-cache kernel, one half in the prefill kernel, where two threads share a
// row. It holds them as fp32 bit patterns in registers.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {
namespace tile {

constexpr int kBN = 128;  // keys per K/V tile
constexpr uint32_t kNegInfBits = 0xff800000u;

// Hides (-inf) the scores outside the visible columns [vlo, vhi] (relative
// to the first of the N held columns); with a zero scale the visible ones
// become 0 (the caller then uses 1 as the multiplier, which keeps -inf * 0
// out of the hidden lanes). Branch-free: one unsigned range test and two
// selects per element.
template <int N = kBN>
__device__ __forceinline__ void mask_cols(uint32_t* r, int vlo, int vhi, bool zero_scale) {
  int lo = max(vlo, 0);
  const int hi = min(vhi, N - 1);
  unsigned span = static_cast<unsigned>(hi - lo);
  if (hi < lo) {  // nothing visible in these columns
    lo = 2 * N;
    span = 0;
  }
  const uint32_t keep = zero_scale ? 0u : 0xffffffffu;
#pragma unroll
  for (int e = 0; e < N; ++e)
    r[e] = static_cast<unsigned>(e - lo) <= span ? (r[e] & keep) : kNegInfBits;
}

// Maximum of the N held scores (four independent max3 chains).
template <int N = kBN>
__device__ __forceinline__ float row_max(const uint32_t* r) {
  static_assert(N % 8 == 0, "columns");
  float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
  for (int e = 0; e < N; e += 8) {
    a0 = ptx::max3(a0, __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
    a1 = ptx::max3(a1, __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
    a2 = ptx::max3(a2, __uint_as_float(r[e + 4]), __uint_as_float(r[e + 5]));
    a3 = ptx::max3(a3, __uint_as_float(r[e + 6]), __uint_as_float(r[e + 7]));
  }
  return ptx::max3(a0, a1, fmaxf(a2, a3));
}

// After tmem_wait_ld(), pass each reduced maximum through an empty asm so
// that no use of it can be scheduled above the wait.
template <int N>
__device__ __forceinline__ void float_fence(float* m) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+f"(m[i]));
}

// Maximum of the four per-32-column maxima of a 128-column tile.
__device__ __forceinline__ float max_of(const float* pm) {
  return ptx::max3(pm[0], pm[1], fmaxf(pm[2], pm[3]));
}

// P = 2^(s * ce + neg_base) for the N held scores (hidden scores are -inf
// and give 0), written as N/2 bf16 pairs over r[0..N/2-1]; returns the fp32
// sum of the (unrounded) P. Pairs of columns use packed FMAs and adds.
template <int N = kBN>
__device__ __forceinline__ float exp2_to_bf16(uint32_t* r, float ce, float neg_base) {
  const uint64_t c2 = ptx::pair(__float_as_uint(ce), __float_as_uint(ce));
  const uint64_t nb2 = ptx::pair(__float_as_uint(neg_base), __float_as_uint(neg_base));
  uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    uint32_t lo, hi;
    ptx::unpair(ptx::fma2(ptx::pair(r[2 * i], r[2 * i + 1]), c2, nb2), lo, hi);
    lo = __float_as_uint(ptx::ex2_approx(__uint_as_float(lo)));
    hi = __float_as_uint(ptx::ex2_approx(__uint_as_float(hi)));
    const uint64_t pp = ptx::pair(lo, hi);
    if ((i & 3) == 0) acc0 = ptx::add2(acc0, pp);
    if ((i & 3) == 1) acc1 = ptx::add2(acc1, pp);
    if ((i & 3) == 2) acc2 = ptx::add2(acc2, pp);
    if ((i & 3) == 3) acc3 = ptx::add2(acc3, pp);
    r[i] = ptx::pack_bf16x2(__uint_as_float(lo), __uint_as_float(hi));
  }
  uint32_t u0, u1;
  ptx::unpair(ptx::add2(ptx::add2(acc0, acc1), ptx::add2(acc2, acc3)), u0, u1);
  return __uint_as_float(u0) + __uint_as_float(u1);
}

// Writes 32 output columns c0 .. c0+31 of one row, times inv_l, as bf16 into
// a staging tile laid out like a TMA box of [rows][64 bf16] with the 128-byte
// swizzle (one such box per 64 columns, box_bytes apart).
__device__ __forceinline__ void stage_bf16_sw128(uint8_t* stage, int box_bytes, int row, int c0,
                                                 const uint32_t* o, float inv_l) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 pk;
    pk.x = ptx::pack_bf16x2(__uint_as_float(o[8 * u + 0]) * inv_l,
                            __uint_as_float(o[8 * u + 1]) * inv_l);
    pk.y = ptx::pack_bf16x2(__uint_as_float(o[8 * u + 2]) * inv_l,
                            __uint_as_float(o[8 * u + 3]) * inv_l);
    pk.z = ptx::pack_bf16x2(__uint_as_float(o[8 * u + 4]) * inv_l,
                            __uint_as_float(o[8 * u + 5]) * inv_l);
    pk.w = ptx::pack_bf16x2(__uint_as_float(o[8 * u + 6]) * inv_l,
                            __uint_as_float(o[8 * u + 7]) * inv_l);
    const int chunk = ((c0 & 63) >> 3) + u;  // 16-byte chunk within the 128-byte row
    const int box = c0 >> 6;
    const int phys = chunk ^ (row & 7);       // 128-byte swizzle
    *reinterpret_cast<uint4*>(stage + box * box_bytes + row * 128 + phys * 16) = pk;
  }
}

// As stage_bf16_sw128 for boxes of [rows][32 bf16] (64-byte rows) with the
// 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3).
// c0 is a multiple of 32: the 32 columns fill one box.
__device__ __forceinline__ void stage_bf16_sw64(uint8_t* stage, int box_bytes, int row, int c0,
                                                const uint32_t* o, float inv_l) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 pk;
    pk.x = ptx::pack_bf16x2(__uint_as_float(o[8 * u + 0]) * inv_l,
                            __uint_as_float(o[8 * u + 1]) * inv_l);
    pk.y = ptx::pack_bf16x2(__uint_as_float(o[8 * u + 2]) * inv_l,
                            __uint_as_float(o[8 * u + 3]) * inv_l);
    pk.z = ptx::pack_bf16x2(__uint_as_float(o[8 * u + 4]) * inv_l,
                            __uint_as_float(o[8 * u + 5]) * inv_l);
    pk.w = ptx::pack_bf16x2(__uint_as_float(o[8 * u + 6]) * inv_l,
                            __uint_as_float(o[8 * u + 7]) * inv_l);
    const int phys = u ^ ((row >> 1) & 3);
    *reinterpret_cast<uint4*>(stage + (c0 >> 5) * box_bytes + row * 64 + phys * 16) = pk;
  }
}

}  // namespace tile
}  // namespace fa
