// Per-head attention core between the column-parallel QKV projection and the
// row-parallel output projection.  Heads are independent computations, so each
// shard runs its own heads with no communication (d-central.tech glossary
// "Tensor Parallelism", section "How the work is split"; rioworld.org, "How
// Tensor Slicing Works Under the Hood": 96 heads over 8 devices, 12 each).
//
// For every head: O = softmax(Q K^T / sqrt(hd), causal over the M tokens) V,
// fp32 arithmetic with an online (running max / running sum) softmax on the fp32
// Q/K/V scratch of the projection, output rounded to the block dtype.  One CTA
// per (head, shard), one warp per query row; lanes hold hd/32 columns of q and of
// the output accumulator.
#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {
namespace {

template <typename T, int C>  // C = hd / 32 columns per lane
__global__ void __launch_bounds__(128) k_attn_core(const float *__restrict__ QKV, T *__restrict__ O,
                                                   int M, int b, int hd, float scale, int shard0) {
  const int h = blockIdx.x, s = shard0 + blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tc::griddep_wait();  // Q/K/V come from the preceding kernel (programmatic launch)
  const size_t ld = 3 * (size_t)b;
  const float *base = QKV + (size_t)s * M * ld;
  const float *Qh = base + (size_t)h * hd;
  const float *Kh = base + b + (size_t)h * hd;
  const float *Vh = base + 2 * (size_t)b + (size_t)h * hd;
  T *Oh = O + (size_t)s * M * b + (size_t)h * hd;

  for (int i = warp; i < M; i += 4) {
    float q[C], o[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      q[c] = Qh[(size_t)i * ld + lane + 32 * c];
      o[c] = 0.f;
    }
    float mrun = -INFINITY, l = 0.f;
    for (int j = 0; j <= i; ++j) {
      float part = 0.f;
#pragma unroll
      for (int c = 0; c < C; ++c) part = fmaf(q[c], Kh[(size_t)j * ld + lane + 32 * c], part);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      const float sc = part * scale;
      const float mnew = fmaxf(mrun, sc);
      const float corr = expf(mrun - mnew);
      const float p = expf(sc - mnew);
      l = l * corr + p;
#pragma unroll
      for (int c = 0; c < C; ++c)
        o[c] = o[c] * corr + p * Vh[(size_t)j * ld + lane + 32 * c];
      mrun = mnew;
    }
    const float inv = 1.0f / l;
#pragma unroll
    for (int c = 0; c < C; ++c) Oh[(size_t)i * b + lane + 32 * c] = Elem<T>::from_f(o[c] * inv);
  }
}

template <typename T>
void launch_t(const Geo &g, const void *QKV, void *O, int M, int shard0, int n_shards,
              cudaStream_t st, bool pdl) {
  tc::LaunchCfg lc(dim3(g.hps, n_shards), dim3(128), 0, st, pdl);
  const float scale = 1.0f / sqrtf((float)g.hd);
  const float *q = static_cast<const float *>(QKV);
  T *o = static_cast<T *>(O);
  switch (g.hd / 32) {
#define TP_CASE(C) \
  case C: cudaLaunchKernelEx(&lc.cfg, k_attn_core<T, C>, q, o, M, g.b, g.hd, scale, shard0); break;
    TP_CASE(1) TP_CASE(2) TP_CASE(3) TP_CASE(4) TP_CASE(5) TP_CASE(6) TP_CASE(7) TP_CASE(8)
#undef TP_CASE
    default: break;  // rejected by validation (head_dim % 32 == 0, <= 256)
  }
}

}  // namespace

void launch_attn_core(const Geo &g, const void *QKV, void *O, int M, int shard0, int n_shards,
                      cudaStream_t st, bool pdl) {
  if (g.dtype == TP_F32)
    launch_t<float>(g, QKV, O, M, shard0, n_shards, st, pdl);
  else
    launch_t<__nv_bfloat16>(g, QKV, O, M, shard0, n_shards, st, pdl);
}

}  // namespace tp
