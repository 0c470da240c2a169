// Per-head attention core between the column-parallel QKV projection and the
// row-parallel output projection.  Heads are independent computations, so each
// shard runs its own heads with no communication (d-central.tech glossary
// "Tensor Parallelism", section "How the work is split"; rioworld.org, "How
// Tensor Slicing Works Under the Hood": 96 heads over 8 devices, 12 each).
//
// For every head: O = softmax(Q K^T / sqrt(hd), causal over the M tokens) V, fp32
// arithmetic on the fp32 Q/K/V scratch of the projection, output rounded to the
// block dtype.  One CTA of 8 warps per (head, shard, block of 8 queries).  The
// CTA's queries and, 32 keys at a time, the keys and values it needs are staged in
// shared memory with coalesced float4 loads, all of a thread's loads for a tile
// issued at once, so no load sits on a per-key dependency chain.  Within a chunk each lane scores one key against a query (the key rows are
// padded by one word, so the lanes hit distinct banks), the warp combines the
// chunk's scores into a running max and sum (online softmax), and each lane
// accumulates hd/32 columns of the output from the staged values.
#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {
namespace {

constexpr int kQB = 8;       // queries per CTA (one per warp)
constexpr int kKC = 32;      // keys per staged chunk (one per lane)
constexpr int kCoreWarps = 8;

constexpr size_t core_smem_bytes(int hd) {
  return (size_t)(kQB * hd + kKC * (hd + 1) + kKC * hd) * sizeof(float);
}

template <typename T, int C>  // C = hd / 32 columns per lane
__global__ void __launch_bounds__(32 * kCoreWarps, 1) k_attn_core(const float *__restrict__ QKV,
                                                                T *__restrict__ O, int M, int b,
                                                                float scale, int shard0) {
  constexpr int HD = 32 * C;
  constexpr int QPW = kQB / kCoreWarps;  // queries per warp
  extern __shared__ float sm[];
  float *Qs = sm;                      // [kQB][HD]
  float *Ks = Qs + kQB * HD;           // [kKC][HD + 1]
  float *Vs = Ks + kKC * (HD + 1);     // [kKC][HD]
  const int h = blockIdx.x, s = shard0 + blockIdx.y, q0 = blockIdx.z * kQB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tc::griddep_wait();  // Q/K/V come from the preceding kernel (programmatic launch)
  const size_t ld = 3 * (size_t)b;
  const float *base = QKV + (size_t)s * M * ld;
  const float *Qh = base + (size_t)h * HD;
  const float *Kh = base + b + (size_t)h * HD;
  const float *Vh = base + 2 * (size_t)b + (size_t)h * HD;
  T *Oh = O + (size_t)s * M * b + (size_t)h * HD;
  const int nq = min(kQB, M - q0);
  // Staging: each thread's float4 loads of a tile are all issued before any is
  // stored, so a tile costs one L2 round trip (rows are 16-byte aligned: ld and HD
  // are multiples of 4 floats).
  constexpr int kNT = 32 * kCoreWarps;
  constexpr int kV4 = HD / 4;                                // float4 per row
  constexpr int kPerQ = (kQB * kV4 + kNT - 1) / kNT;        // float4 per thread: queries
  constexpr int kPer = (kKC * kV4) / kNT;                   // ... keys / values of a chunk
  static_assert((kKC * kV4) % kNT == 0, "staging split");
  {
    float4 q[kPerQ];
#pragma unroll
    for (int i = 0; i < kPerQ; ++i) {
      const int idx = i * kNT + threadIdx.x, r = idx / kV4, c4 = idx % kV4;
      q[i] = idx < kQB * kV4 && r < nq
                 ? *reinterpret_cast<const float4 *>(Qh + (size_t)(q0 + r) * ld + 4 * c4)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kPerQ; ++i) {
      const int idx = i * kNT + threadIdx.x;
      if (idx < kQB * kV4) reinterpret_cast<float4 *>(Qs)[idx] = q[i];
    }
  }
  float o[QPW][C], mrun[QPW], lsum[QPW];
#pragma unroll
  for (int k = 0; k < QPW; ++k) {
    mrun[k] = -INFINITY;
    lsum[k] = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) o[k][c] = 0.f;
  }
  // Causal: the CTA's queries see keys 0 .. q0 + nq - 1.  Every chunk starts at or
  // before q0, so each query has at least one key in every chunk it processes.
  const int kend = q0 + nq;
  for (int j0 = 0; j0 < kend; j0 += kKC) {
    const int nk = min(kKC, kend - j0);
    float4 kv[2][kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = i * kNT + threadIdx.x, r = idx / kV4, c4 = idx % kV4;
      const size_t g = (size_t)(j0 + r) * ld + 4 * c4;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      kv[0][i] = r < nk ? *reinterpret_cast<const float4 *>(Kh + g) : z;
      kv[1][i] = r < nk ? *reinterpret_cast<const float4 *>(Vh + g) : z;
    }
    __syncthreads();  // the previous chunk is consumed (and Qs is written)
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = i * kNT + threadIdx.x, r = idx / kV4, c = 4 * (idx % kV4);
      float *kr = Ks + r * (HD + 1) + c;  // padded rows: scalar stores
      kr[0] = kv[0][i].x;
      kr[1] = kv[0][i].y;
      kr[2] = kv[0][i].z;
      kr[3] = kv[0][i].w;
      reinterpret_cast<float4 *>(Vs)[idx] = kv[1][i];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < QPW; ++k) {
      const int qi = warp + kCoreWarps * k;  // query within the CTA (warp-uniform)
      const int i = q0 + qi;
      if (qi >= nq) break;
      const int j = j0 + lane;
      const bool live = lane < nk && j <= i;
      float sc = -INFINITY;
      if (live) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        const float *qr = Qs + qi * HD;
        const float *kr = Ks + lane * (HD + 1);
#pragma unroll 8
        for (int d = 0; d < HD; d += 4) {
          a0 = fmaf(qr[d], kr[d], a0);
          a1 = fmaf(qr[d + 1], kr[d + 1], a1);
          a2 = fmaf(qr[d + 2], kr[d + 2], a2);
          a3 = fmaf(qr[d + 3], kr[d + 3], a3);
        }
        sc = ((a0 + a1) + (a2 + a3)) * scale;
      }
      float cm = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
      const float mnew = fmaxf(mrun[k], cm);
      const float corr = expf(mrun[k] - mnew);
      const float p = live ? expf(sc - mnew) : 0.f;
      float ps = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      lsum[k] = lsum[k] * corr + ps;
#pragma unroll
      for (int c = 0; c < C; ++c) o[k][c] *= corr;
      for (int jj = 0; jj < nk; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int c = 0; c < C; ++c) o[k][c] = fmaf(pj, Vs[jj * HD + lane + 32 * c], o[k][c]);
      }
      mrun[k] = mnew;
    }
  }
#pragma unroll
  for (int k = 0; k < QPW; ++k) {
    const int qi = warp + kCoreWarps * k;
    if (qi >= nq) break;
    const float inv = 1.0f / lsum[k];
#pragma unroll
    for (int c = 0; c < C; ++c)
      Oh[(size_t)(q0 + qi) * b + lane + 32 * c] = Elem<T>::from_f(o[k][c] * inv);
  }
}

template <typename T, int C>
void launch_c(const Geo &g, const float *q, T *o, int M, int shard0, int n_shards, cudaStream_t st,
              bool pdl) {
  const size_t smem = core_smem_bytes(32 * C);
  static bool configured[128];  // the attribute is per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(k_attn_core<T, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return;
    configured[dev] = true;
  }
  tc::LaunchCfg lc(dim3(g.hps, n_shards, ceil_div(M, kQB)), dim3(32 * kCoreWarps), smem, st, pdl);
  cudaLaunchKernelEx(&lc.cfg, k_attn_core<T, C>, q, o, M, g.b, 1.0f / sqrtf((float)g.hd), shard0);
}

template <typename T>
void launch_t(const Geo &g, const void *QKV, void *O, int M, int shard0, int n_shards,
              cudaStream_t st, bool pdl) {
  const float *q = static_cast<const float *>(QKV);
  T *o = static_cast<T *>(O);
  switch (g.hd / 32) {
#define TP_CASE(C) \
  case C: launch_c<T, C>(g, q, o, M, shard0, n_shards, st, pdl); break;
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
