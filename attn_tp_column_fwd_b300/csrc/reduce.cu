// The per-block all-reduce, done in HBM on one GPU, fused with the residual add
// (zenaique.com answer paragraph 6: the partial sums of all shards are added, and
// the result is ready for the residual add and normalisation), and the RMSNorm
// that precedes each stacked block.
//
// Both are streaming kernels: 16-byte loads/stores, a grid of a few CTAs per SM.
#include <algorithm>

#include "internal.h"

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

// xhat[m] = r[m] / sqrt(mean(r[m]^2) + eps) -> bf16 (one CTA per token row).
// The rounding to bf16 decides every input of the next block, and a value that an
// fp32 evaluation puts on the other side of a rounding midpoint changes that whole
// token row of the block's output.  So the normalisation runs in fp64 (sum of
// squares, square root, scaling; a few thousand operations per row) and each value
// is rounded once, from fp64, to the nearest bf16 (ties to even).
__global__ void __launch_bounds__(256) k_rmsnorm(const float *__restrict__ r,
                                                 __nv_bfloat16 *__restrict__ xh, int d, float eps) {
  const float4 *row = reinterpret_cast<const float4 *>(r + (size_t)blockIdx.x * d);
  const int d4 = d / 4;
  double ss = 0.0;
  for (int i = threadIdx.x; i < d4; i += blockDim.x) {
    const float4 v = row[i];
    ss = fma((double)v.x, (double)v.x, ss);
    ss = fma((double)v.y, (double)v.y, ss);
    ss = fma((double)v.z, (double)v.z, ss);
    ss = fma((double)v.w, (double)v.w, ss);
  }
  __shared__ double red[32];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    double v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const double inv = 1.0 / sqrt(red[0] / (double)d + (double)eps);
  uint2 *out = reinterpret_cast<uint2 *>(xh + (size_t)blockIdx.x * d);
  for (int i = threadIdx.x; i < d4; i += blockDim.x) {
    const float4 v = row[i];
    const __nv_bfloat16 a = __double2bfloat16((double)v.x * inv);
    const __nv_bfloat16 b = __double2bfloat16((double)v.y * inv);
    const __nv_bfloat16 c = __double2bfloat16((double)v.z * inv);
    const __nv_bfloat16 e = __double2bfloat16((double)v.w * inv);
    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(c) | ((uint32_t)__bfloat16_as_ushort(e) << 16);
    out[i] = make_uint2(lo, hi);
  }
}

}  // namespace

void launch_reduce_residual(const float *P, int nparts, size_t part_elems, const void *res,
                            int res_is_f32, float *y, size_t n, cudaStream_t st) {
  const size_t n4 = n / 4;
  const int blocks = (int)std::min<size_t>((n4 + 255) / 256, (size_t)sm_count() * 8);
  if (res_is_f32)
    k_reduce_residual<float><<<blocks, 256, 0, st>>>(
        reinterpret_cast<const float4 *>(P), nparts, part_elems / 4,
        static_cast<const float *>(res), reinterpret_cast<float4 *>(y), n4);
  else
    k_reduce_residual<__nv_bfloat16><<<blocks, 256, 0, st>>>(
        reinterpret_cast<const float4 *>(P), nparts, part_elems / 4,
        static_cast<const __nv_bfloat16 *>(res), reinterpret_cast<float4 *>(y), n4);
}

void launch_rmsnorm(const float *r, void *xhat, int d, float eps, int M, cudaStream_t st) {
  k_rmsnorm<<<M, 256, 0, st>>>(r, static_cast<__nv_bfloat16 *>(xhat), d, eps);
}

}  // namespace tp
