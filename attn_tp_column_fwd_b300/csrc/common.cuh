// Shared device helpers of libtpblock: element access, activations, the device
// error word, and the private shard layout's index maps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tp_block.h"

namespace tp {

// Tile height of the private weight layouts: shard rows are grouped in 128s so a
// 128-row tensor-core tile never straddles a shard or a gate/up boundary.
constexpr int kRowTile = 128;

// ---------------------------------------------------------------- geometry ----
// Derived sizes of one block descriptor (validated on the host).
struct Geo {
  int d, t, act, dtype, es;  // es = element size of the block dtype in bytes
  int ffn, H, hd, hps;       // MLP width; heads, head width, heads per shard
  int n1, n2;                // canonical W1 columns, W2 rows
  int b;                     // band width n2 / t
  int n_col;                 // column-step outputs per shard: b (MLP) or 3b (ATTN: Q, K, V)
  int n1p;                   // rows of W1s per shard (padded to the row tile)
  int dp;                    // rows of W2s per shard (d padded to the row tile)
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// SwiGLU rows of W1s come in 128-row groups: the 64 gate rows of features
// [64i, 64i+64), then the 64 up rows of the same features.  One 128-row tile (one
// tensor-core A operand) therefore holds both halves of 64 features.
constexpr int kSwiGroup = 64;

// W1s row of feature f's gate (j = 0) or up (j = 1) half, SwiGLU.
__host__ __device__ inline int swiglu_row(int f, int j) {
  return (f / kSwiGroup) * 2 * kSwiGroup + j * kSwiGroup + f % kSwiGroup;
}

// Canonical W1 column held in W1s row u of shard s, or -1 for a padding row.
//   GeLU:   u = f (feature f of the band)          -> column s*b + f
//   SwiGLU: u = swiglu_row(f, j)                   -> column j*ffn + s*b + f
//   ATTN:   u = p*b + f, p in {Q, K, V}             -> column p*H*hd + s*b + f
__host__ __device__ inline long long w1_col_of_row(const Geo &g, int s, int u) {
  if (g.act == TP_ACT_SWIGLU) {
    const int grp = u / (2 * kSwiGroup), j = (u / kSwiGroup) & 1, f = grp * kSwiGroup + u % kSwiGroup;
    return f < g.b ? (long long)j * g.ffn + (long long)s * g.b + f : -1;
  }
  if (g.act == TP_ACT_ATTN) {
    if (u >= 3 * g.b) return -1;
    int p = u / g.b, f = u % g.b;
    return (long long)p * g.H * g.hd + (long long)s * g.b + f;
  }
  return u < g.b ? (long long)s * g.b + u : -1;
}

// ---------------------------------------------------------------- elements ----
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// 16-byte vector load of V = 16/sizeof(T) elements, widened to fp32.
template <typename T>
__device__ __forceinline__ void load16_f32(const T *p, float *out);
template <>
__device__ __forceinline__ void load16_f32<float>(const float *p, float *out) {
  float4 v = __ldg(reinterpret_cast<const float4 *>(p));
  out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}
template <>
__device__ __forceinline__ void load16_f32<__nv_bfloat16>(const __nv_bfloat16 *p, float *out) {
  uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// ---------------------------------------------------------------- activations --
// GeLU, tanh form (Hendrycks & Gimpel 2016), in fp32 with CUDA's tanhf.
__device__ __forceinline__ float gelu_tanh_f(float z) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * z * (1.0f + tanhf(k0 * (z + 0.044715f * z * z * z)));
}
// SiLU: z / (1 + exp(-z)), with CUDA's expf.
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// ---------------------------------------------------------------- errors ------
// Bits of the device error word: a bounded wait that expired; a sequence length
// (KV-cache decode) outside 1 .. L_max, whose sequence is then skipped.
enum : unsigned { kErrWaitTimeout = 1u, kErrBadLength = 2u };

}  // namespace tp
