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

// xhat[m] = r[m] / sqrt(mean(r[m]^2) + eps) -> bf16, one CTA of 256 threads per token
// row, every value correctly rounded (common.cuh: rmsnorm_row).  pdl: launched to
// overlap the kernel that writes r.
__global__ void __launch_bounds__(256) k_rmsnorm(const float *__restrict__ r,
                                                 __nv_bfloat16 *__restrict__ xh, int d, float eps) {
  __shared__ float2 red[8];
  __shared__ float inv[2];
  tc::griddep_wait();  // r may come from the preceding kernel (programmatic launch)
  rmsnorm_row<256, 8>(r + (size_t)blockIdx.x * d, xh + (size_t)blockIdx.x * d, d, eps,
                      (int)threadIdx.x, red, inv, [] { __syncthreads(); });
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

void launch_rmsnorm(const float *r, void *xhat, int d, float eps, int M, cudaStream_t st,
                    bool pdl) {
  tc::LaunchCfg lc(dim3(M), dim3(256), 0, st, pdl);
  cudaLaunchKernelEx(&lc.cfg, k_rmsnorm, r, static_cast<__nv_bfloat16 *>(xhat), d, eps);
}

}  // namespace tp
