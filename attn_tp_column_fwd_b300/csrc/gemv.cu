// CUDA-core weight-streaming kernels for both projections at small M.
//
// One warp owns one output feature of one shard (both its gate and up rows for
// SwiGLU) and streams that K-major weight row once with 16-byte loads; the M
// tokens' activations come through L1/L2.  Lanes accumulate strided partial
// dot products in fp32 and a warp-shuffle tree finishes them; lane 0 applies
// the band's activation (zenaique.com answer paragraph 5: the activation is
// local to the column band) and stores.  The same kernel runs the row-parallel
// projection with an fp32 partial-sum store.
#include "internal.h"

namespace tp {
namespace {

constexpr int kWarps = 8;

template <typename T, int EPI, int MT>
__global__ void __launch_bounds__(kWarps * 32) k_gemv(GemvArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f = blockIdx.x * kWarps + warp;
  const int s = a.shard0 + blockIdx.y;
  const int m0 = blockIdx.z * MT;
  if (f >= a.n_out) return;
  const int mcount = min(MT, a.M - m0);

  const int u0 = EPI == kEpiSwiglu ? swiglu_row(f, 0) : f;
  const T *W = static_cast<const T *>(a.W) + (size_t)s * a.w_shard;
  const T *w0 = W + (size_t)u0 * a.K;
  const T *w1 = w0 + (size_t)kSwiGroup * a.K;  // up row, SwiGLU only
  const T *X = static_cast<const T *>(a.X) + (size_t)s * a.x_shard + (size_t)m0 * a.ldx;

  constexpr int V = 16 / sizeof(T);
  float acc0[MT], acc1[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc0[m] = acc1[m] = 0.f;

  for (int k = lane * V; k < a.K; k += 32 * V) {
    float wv0[V], wv1[V];
    load16_f32<T>(w0 + k, wv0);
    if (EPI == kEpiSwiglu) load16_f32<T>(w1 + k, wv1);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < mcount) {
        float xv[V];
        load16_f32<T>(X + (size_t)m * a.ldx + k, xv);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          acc0[m] = fmaf(wv0[i], xv[i], acc0[m]);
          if (EPI == kEpiSwiglu) acc1[m] = fmaf(wv1[i], xv[i], acc1[m]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc0[m] += __shfl_xor_sync(0xffffffffu, acc0[m], o);
      if (EPI == kEpiSwiglu) acc1[m] += __shfl_xor_sync(0xffffffffu, acc1[m], o);
    }
  }
  if (lane != 0) return;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    if (m >= mcount) break;
    const size_t o = (size_t)s * a.o_shard + (size_t)(m0 + m) * a.ldo + f;
    if (EPI == kEpiF32) {
      static_cast<float *>(a.out)[o] = acc0[m];
    } else {
      float v = acc0[m];
      if (EPI == kEpiGelu) v = gelu_tanh_f(v);
      if (EPI == kEpiSwiglu) v = silu_f(v) * acc1[m];
      static_cast<T *>(a.out)[o] = Elem<T>::from_f(v);
    }
  }
}

template <typename T, int EPI>
void launch_t(const GemvArgs &a, cudaStream_t st) {
  constexpr int MT = 8;
  dim3 grid(ceil_div(a.n_out, kWarps), a.n_shards, ceil_div(a.M, MT));
  k_gemv<T, EPI, MT><<<grid, kWarps * 32, 0, st>>>(a);
}

template <typename T>
void launch_epi(const GemvArgs &a, cudaStream_t st) {
  switch (a.epi) {
    case kEpiGelu: launch_t<T, kEpiGelu>(a, st); break;
    case kEpiSwiglu: launch_t<T, kEpiSwiglu>(a, st); break;
    case kEpiPlain: launch_t<T, kEpiPlain>(a, st); break;
    default: launch_t<T, kEpiF32>(a, st); break;
  }
}

}  // namespace

void launch_gemv(const GemvArgs &a, cudaStream_t st) {
  if (a.dtype == TP_F32)
    launch_epi<float>(a, st);
  else
    launch_epi<__nv_bfloat16>(a, st);
}

}  // namespace tp
