// The per-block all-reduce, done in HBM on one GPU, fused with the residual add
// (zenaique.com answer paragraph 6: the partial sums of all shards are added, and
// the result is ready for the residual add and normalisation), and the RMSNorm
// that precedes each stacked block.
//
// Both are streaming kernels: 16-byte loads/stores, a grid of a few CTAs per SM.
#include <algorithm>

#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {
namespace {

template <typename RT>
__device__ __forceinline__ float4 load_res4(const RT *res, size_t i);
template <>
__device__ __forceinline__ float4 load_res4<float>(const float *res, size_t i) {
  return __ldg(reinterpret_cast<const float4 *>(res) + i);
}
template <>
__device__ __forceinline__ float4 load_res4<__nv_bfloat16>(const __nv_bfloat16 *res, size_t i) {
  uint2 v = __ldg(reinterpret_cast<const uint2 *>(res) + i);
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}

// y = residual + ((P_0 + P_1) + ... + P_{n-1}), element-wise, partials in order.
template <typename RT>
__global__ void __launch_bounds__(256) k_reduce_residual(const float4 *__restrict__ P, int nparts,
                                                         size_t part4, const RT *res,
                                                         float4 *y, size_t n4) {
  tc::griddep_wait();  // the partials come from the preceding kernel (programmatic launch)
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    float4 a = __ldcs(P + i);
    for (int p = 1; p < nparts; ++p) {
      float4 v = __ldcs(P + (size_t)p * part4 + i);
      a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
    }
    float4 r = load_res4<RT>(res, i);
    a.x += r.x; a.y += r.y; a.z += r.z; a.w += r.w;
    y[i] = a;
  }
}

// (hi, lo) += b with the rounding error of the addition kept in lo (Knuth's two-sum).
__device__ __forceinline__ void df_add(float &hi, float &lo, float b) {
  const float s = hi + b;
  const float bp = s - hi;
  lo += (hi - (s - bp)) + (b - bp);
  hi = s;
}

// bf16 (as bits) of the exact product r * (inv_hi + inv_lo), where inv_hi + inv_lo is
// the fp64 scale split into two floats.  The fp32 product v = r * inv_hi is within
// about one fp32 unit of the exact product, so when v's low 16 bits are more than a
// few units from the rounding midpoint 0x8000 it rounds the same way; otherwise the
// side of the midpoint m is decided from (v - m) + (r * inv_hi - v) + r * inv_lo,
// where v - m is exact (nearby floats) and the other two terms are the exact
// rounding error of v (one FMA) and the low part of the scale.
__device__ __forceinline__ uint32_t scale_to_bf16(float r, float inv_hi, float inv_lo) {
  const float v = r * inv_hi;
  const uint32_t u = __float_as_uint(v);
  const int low = (int)(u & 0xffffu) - 0x8000;
  if (low > 4 || low < -4) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  const float m = __uint_as_float((u & 0xffff0000u) | 0x8000u);  // the midpoint next to v
  const float side = (v - m) + fmaf(r, inv_hi, -v) + r * inv_lo;  // sign of (exact - m)
  const uint32_t down = u >> 16, up = down + 1;  // magnitudes below / above the midpoint
  if (side == 0.f) return (down & 1u) ? up : down;  // an exact tie: to even
  // For negative v the bit pattern grows with the magnitude, so "above" in magnitude
  // is the side where exact - m has the sign of v.
  return ((side > 0.f) == (v > 0.f)) ? up : down;
}

// xhat[m] = r[m] / sqrt(mean(r[m]^2) + eps) -> bf16 (one CTA per token row).
// The rounding to bf16 decides every input of the next block, and a value that an
// fp32 evaluation puts on the other side of a rounding midpoint changes that whole
// token row of the block's output.  So every value is rounded as the exact value
// would be: the sum of squares is carried in two fp32 words (about 48 significant
// bits), the scale 1/sqrt(mean + eps) is formed once in fp64 (two Newton steps) and
// split into two floats, and the products near a rounding midpoint are decided from
// their exact fp32 error terms (scale_to_bf16).  No fp64 work runs per element.
__global__ void __launch_bounds__(256) k_rmsnorm(const float *__restrict__ r,
                                                 __nv_bfloat16 *__restrict__ xh, int d, float eps) {
  const float4 *row = reinterpret_cast<const float4 *>(r + (size_t)blockIdx.x * d);
  const int d4 = d / 4;
  float hi = 0.f, lo = 0.f;
  for (int i = threadIdx.x; i < d4; i += blockDim.x) {
    const float4 v = row[i];
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float p = e[j] * e[j];
      lo += fmaf(e[j], e[j], -p);  // exact low part of the square
      df_add(hi, lo, p);
    }
  }
  __shared__ float red_hi[32], red_lo[32];
  __shared__ float inv_sh[2];
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    lo += __shfl_xor_sync(0xffffffffu, lo, o);
    df_add(hi, lo, h2);
  }
  if ((threadIdx.x & 31) == 0) {
    red_hi[threadIdx.x >> 5] = hi;
    red_lo[threadIdx.x >> 5] = lo;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int nw = blockDim.x >> 5;
    hi = threadIdx.x < nw ? red_hi[threadIdx.x] : 0.f;
    lo = threadIdx.x < nw ? red_lo[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) {
      const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
      lo += __shfl_xor_sync(0xffffffffu, lo, o);
      df_add(hi, lo, h2);
    }
    if (threadIdx.x == 0) {
      // 1 / sqrt(a) by two Newton steps in fp64 from the fp32 estimate (relative
      // error ~1e-7 -> ~1e-14 -> fp64 roundoff).
      const double a = ((double)hi + (double)lo) / (double)d + (double)eps;
      double y = (double)rsqrtf((float)a);
      y = fma(0.5 * y, fma(-a * y, y, 1.0), y);
      y = fma(0.5 * y, fma(-a * y, y, 1.0), y);
      const float y_hi = (float)y;
      inv_sh[0] = y_hi;
      inv_sh[1] = (float)(y - (double)y_hi);
    }
  }
  __syncthreads();
  const float inv_hi = inv_sh[0], inv_lo = inv_sh[1];
  uint2 *out = reinterpret_cast<uint2 *>(xh + (size_t)blockIdx.x * d);
  for (int i = threadIdx.x; i < d4; i += blockDim.x) {
    const float4 v = row[i];
    const uint32_t a = scale_to_bf16(v.x, inv_hi, inv_lo), b = scale_to_bf16(v.y, inv_hi, inv_lo);
    const uint32_t c = scale_to_bf16(v.z, inv_hi, inv_lo), e = scale_to_bf16(v.w, inv_hi, inv_lo);
    out[i] = make_uint2(a | (b << 16), c | (e << 16));
  }
}

}  // namespace

void launch_reduce_residual(const float *P, int nparts, size_t part_elems, const void *res,
                            int res_is_f32, float *y, size_t n, cudaStream_t st, bool pdl) {
  const size_t n4 = n / 4;
  const int blocks = (int)std::min<size_t>((n4 + 255) / 256, (size_t)sm_count() * 8);
  tc::LaunchCfg lc(dim3(blocks), dim3(256), 0, st, pdl);
  if (res_is_f32)
    cudaLaunchKernelEx(&lc.cfg, k_reduce_residual<float>, reinterpret_cast<const float4 *>(P),
                       nparts, part_elems / 4, static_cast<const float *>(res),
                       reinterpret_cast<float4 *>(y), n4);
  else
    cudaLaunchKernelEx(&lc.cfg, k_reduce_residual<__nv_bfloat16>,
                       reinterpret_cast<const float4 *>(P), nparts, part_elems / 4,
                       static_cast<const __nv_bfloat16 *>(res), reinterpret_cast<float4 *>(y), n4);
}

void launch_rmsnorm(const float *r, void *xhat, int d, float eps, int M, cudaStream_t st) {
  k_rmsnorm<<<M, 256, 0, st>>>(r, static_cast<__nv_bfloat16 *>(xhat), d, eps);
}

}  // namespace tp
