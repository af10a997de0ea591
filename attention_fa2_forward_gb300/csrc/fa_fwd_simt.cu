// fa_fwd_simt.cu -- fp32 fused attention forward on the CUDA cores.
//
// Same operation as the tensor-core path (MAX API page "FlashAttentionGPU",
// `execute` Steps -1 to 4) for fp32 tensors. fp32 FMA keeps the scores
// exact to fp32 rounding (a TF32 tensor-core product would not), so the
// result stays within 1e-4 of the fp64 definition.
//
// One warp per query row, four rows per CTA; the CTA streams 32-key K/V
// tiles through shared memory; lane j scores key j of the tile, the warp
// keeps the online-softmax state (running max m, running sum l) of the
// FlashAttention-2 loop (tiny_flash_attn.py page, flash_attn_v2), and each
// lane accumulates D/32 output columns. Exponentials use the accurate expf.
#include <cmath>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kRows = 4;   // query rows per CTA (one warp each)
constexpr int kKeys = 32;  // keys per tile (one per lane)

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D>
__global__ void __launch_bounds__(kRows * 32)
    fa_fwd_f32_simt_kernel(const float* __restrict__ q, const float* __restrict__ k,
                           const float* __restrict__ v, float* __restrict__ out,
                           const FwdProblem p, BshdStrides sq, BshdStrides sk, BshdStrides sv,
                           BshdStrides so) {
  constexpr int kPerLane = D / 32;
  __shared__ float sK[kKeys][D + 1];
  __shared__ float sV[kKeys][D];
  __shared__ float sQ[kRows][D];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int hk = h / (p.H / p.Hkv);
  const int r0 = blockIdx.x * kRows;
  const int i = r0 + warp;
  const bool row_valid = i < p.S;

  for (int d = lane; d < D; d += 32)
    sQ[warp][d] = row_valid ? q[b * sq.b + i * sq.s + h * sq.h + d] : 0.f;

  // Keys any row of this CTA may see, and the ones row i sees.
  const int r_last = min(r0 + kRows, p.S) - 1;
  const int kv_begin = p.window > 0 ? max(0, r0 - p.window + 1) : 0;
  const int kv_end =
      p.causal ? r_last + 1 : (p.window > 0 ? min(p.S, r_last + p.window) : p.S);
  const int vis_lo = p.window > 0 ? i - p.window + 1 : 0;
  const int vis_hi =
      p.causal ? min(i, p.S - 1) : (p.window > 0 ? min(i + p.window - 1, p.S - 1) : p.S - 1);

  float m = -INFINITY, l = 0.f;
  float o[kPerLane];
#pragma unroll
  for (int u = 0; u < kPerLane; ++u) o[u] = 0.f;

  for (int k0 = kv_begin; k0 < kv_end; k0 += kKeys) {
    __syncthreads();
    for (int e = threadIdx.x; e < kKeys * D; e += kRows * 32) {
      const int kr = e / D, d = e % D;
      const int key = k0 + kr;
      float kval = 0.f, vval = 0.f;
      if (key < kv_end) {
        kval = k[b * sk.b + key * sk.s + hk * sk.h + d];
        vval = v[b * sv.b + key * sv.s + hk * sv.h + d];
      }
      sK[kr][d] = kval;
      sV[kr][d] = vval;
    }
    __syncthreads();

    const int key = k0 + lane;
    const bool vis = row_valid && key < kv_end && key >= vis_lo && key <= vis_hi;
    float s = -INFINITY;
    if (vis) {
      float dot = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) dot = fmaf(sQ[warp][d], sK[lane][d], dot);
      s = dot * p.scale;
    }
    const float m_new = fmaxf(m, warp_max(s));
    if (m_new == -INFINITY) continue;  // nothing visible to this row yet
    const float alpha = m == -INFINITY ? 0.f : expf(m - m_new);
    const float pj = vis ? expf(s - m_new) : 0.f;
    l = l * alpha + warp_sum(pj);
#pragma unroll
    for (int u = 0; u < kPerLane; ++u) o[u] *= alpha;
    for (int jj = 0; jj < kKeys; ++jj) {
      const float pb = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
      for (int u = 0; u < kPerLane; ++u) o[u] = fmaf(pb, sV[jj][lane + 32 * u], o[u]);
    }
    m = m_new;
  }

  if (row_valid) {
    const float inv_l = 1.f / l;
    float* orow = out + (b * so.b + i * so.s + h * so.h);
#pragma unroll
    for (int u = 0; u < kPerLane; ++u) orow[lane + 32 * u] = o[u] * inv_l;
    if (p.lse != nullptr && lane == 0)
      p.lse[(static_cast<size_t>(b) * p.H + h) * p.S + i] = m + logf(l);
  }
}

template <int D>
cudaError_t launch_d(const FwdProblem& p, float* out, const float* q, const float* k,
                     const float* v, cudaStream_t stream) {
  const dim3 grid((p.S + kRows - 1) / kRows, p.H, p.B);
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidConfiguration;
  fa_fwd_f32_simt_kernel<D><<<grid, kRows * 32, 0, stream>>>(
      q, k, v, out, p, resolve_strides(p.sq, p.S, p.H, D), resolve_strides(p.sk, p.S, p.Hkv, D),
      resolve_strides(p.sv, p.S, p.Hkv, D), resolve_strides(p.so, p.S, p.H, D));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32_simt(const FwdProblem& p, float* out, const float* q, const float* k,
                                const float* v, cudaStream_t stream) {
  switch (p.D) {
    case 32: return launch_d<32>(p, out, q, k, v, stream);
    case 64: return launch_d<64>(p, out, q, k, v, stream);
    case 96: return launch_d<96>(p, out, q, k, v, stream);
    case 128: return launch_d<128>(p, out, q, k, v, stream);
    default: return cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
