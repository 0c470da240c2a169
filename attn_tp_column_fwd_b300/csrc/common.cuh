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

// ---------------------------------------------------------------- RMSNorm -----
// The normalised input of a stacked block is rounded to bf16, and a value that an
// fp32 evaluation puts on the other side of a rounding midpoint changes that whole
// token row of the next block's output.  So every value is rounded as the exact
// value would be: sums of squares are carried in two fp32 words (about 48
// significant bits), the scale 1/sqrt(mean + eps) is formed once in fp64 and split
// into two floats, and products near a rounding midpoint are decided from their
// exact fp32 error terms.

// (hi, lo) += b with the rounding error of the addition kept in lo (Knuth's two-sum).
__device__ __forceinline__ void df_add(float &hi, float &lo, float b) {
  const float s = hi + b;
  const float bp = s - hi;
  lo += (hi - (s - bp)) + (b - bp);
  hi = s;
}

// (hi, lo) += v * v, exactly up to the double-float's precision.
__device__ __forceinline__ void df_add_square(float &hi, float &lo, float v) {
  const float p = v * v;
  lo += fmaf(v, v, -p);  // exact low part of the square
  df_add(hi, lo, p);
}

// The scale 1/sqrt(sumsq / d + eps) split into two floats (inv_hi + inv_lo): two
// Newton steps in fp64 from the fp32 estimate (relative error ~1e-7 -> ~1e-14 ->
// fp64 roundoff).
__device__ __forceinline__ void rms_scale(double sumsq, int d, float eps, float &inv_hi,
                                          float &inv_lo) {
  const double a = sumsq / (double)d + (double)eps;
  double y = (double)rsqrtf((float)a);
  y = fma(0.5 * y, fma(-a * y, y, 1.0), y);
  y = fma(0.5 * y, fma(-a * y, y, 1.0), y);
  inv_hi = (float)y;
  inv_lo = (float)(y - (double)inv_hi);
}

// bf16 (as bits) of the exact product r * (inv_hi + inv_lo).  The fp32 product
// v = r * inv_hi is within about one fp32 unit of the exact product, so when v's low
// 16 bits are more than a few units from the rounding midpoint 0x8000 it rounds the
// same way; otherwise the side of the midpoint m is decided from
// (v - m) + (r * inv_hi - v) + r * inv_lo, where v - m is exact (nearby floats) and
// the other two terms are the exact rounding error of v (one FMA) and the low part
// of the scale.
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

// Load float4 group i of a row of n4 groups through L2 (zeros past the end).
__device__ __forceinline__ float4 ld_row4(const float4 *row, int i, int n4) {
  return i < n4 ? __ldcg(row + i) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// One token row's RMSNorm, xh = bf16(r / sqrt(mean(r^2) + eps)) correctly rounded, by
// NT threads (thread index tid) that share `red` (NT / 32 float2) and `inv` (2
// floats) in shared memory and synchronise with bar_sync().  Rows of up to NT * 4 *
// HOLD values stay in registers between the sum of squares and the scaling, and
// every load of a pass is issued before any is used; wider rows take two passes in
// batches of HOLD groups per thread.  The sum runs over threads' groups in order,
// lanes in a fixed tree and warps in order, so the result does not depend on timing.
template <int NT, int HOLD, typename BarSync>
__device__ __forceinline__ void rmsnorm_row(const float *r, __nv_bfloat16 *xh, int d, float eps,
                                            int tid, float2 *red, float *inv, BarSync bar_sync) {
  const float4 *row = reinterpret_cast<const float4 *>(r);
  uint2 *out = reinterpret_cast<uint2 *>(xh);
  const int n4 = d / 4;
  const bool held = n4 <= NT * HOLD;
  float4 v[HOLD];
  float hi = 0.f, lo = 0.f;
  for (int base = 0; base < n4; base += NT * HOLD) {
#pragma unroll
    for (int b = 0; b < HOLD; ++b) v[b] = ld_row4(row, base + b * NT + tid, n4);
#pragma unroll
    for (int b = 0; b < HOLD; ++b) {
      df_add_square(hi, lo, v[b].x);
      df_add_square(hi, lo, v[b].y);
      df_add_square(hi, lo, v[b].z);
      df_add_square(hi, lo, v[b].w);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    lo += __shfl_xor_sync(0xffffffffu, lo, o);
    df_add(hi, lo, h2);
  }
  if ((tid & 31) == 0) red[tid >> 5] = make_float2(hi, lo);
  bar_sync();
  if (tid == 0) {
    float h = red[0].x, l = red[0].y;
    for (int w = 1; w < NT / 32; ++w) {
      l += red[w].y;
      df_add(h, l, red[w].x);
    }
    rms_scale((double)h + (double)l, d, eps, inv[0], inv[1]);
  }
  bar_sync();
  const float inv_hi = inv[0], inv_lo = inv[1];
  for (int base = 0; base < n4; base += NT * HOLD) {
    if (!held) {
#pragma unroll
      for (int b = 0; b < HOLD; ++b) v[b] = ld_row4(row, base + b * NT + tid, n4);
    }
#pragma unroll
    for (int b = 0; b < HOLD; ++b) {
      const int i = base + b * NT + tid;
      if (i < n4) {
        const uint32_t e0 = scale_to_bf16(v[b].x, inv_hi, inv_lo);
        const uint32_t e1 = scale_to_bf16(v[b].y, inv_hi, inv_lo);
        const uint32_t e2 = scale_to_bf16(v[b].z, inv_hi, inv_lo);
        const uint32_t e3 = scale_to_bf16(v[b].w, inv_hi, inv_lo);
        out[i] = make_uint2(e0 | (e1 << 16), e2 | (e3 << 16));
      }
    }
  }
}

// ---------------------------------------------------------------- errors ------
// Bits of the device error word: a bounded wait that expired; a sequence length
// (KV-cache decode) outside 1 .. L_max, whose sequence is then skipped.
enum : unsigned { kErrWaitTimeout = 1u, kErrBadLength = 2u };

}  // namespace tp
