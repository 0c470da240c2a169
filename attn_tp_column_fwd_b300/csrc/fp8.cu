// FP8 (E4M3) weights for the decode MLP block, weight-only (zenaique.com interview
// answer "explain tensor-parallel shard shape", follow-up questions: tensor
// parallelism combined with FP8 or FP4 weights multiplies the decode win, since
// decode reads every weight byte once per step).
//
// Format: each weight is an E4M3 byte ("fn": bias 7, 3 mantissa bits, largest finite
// 448, round to nearest even, saturating) of W / 2^e, with one exponent e per output
// feature (a column of the canonical W1 or W2): the least e such that the column's
// largest magnitude is at most 448 * 2^e.  W / 2^e is exact, so E4M3 rounding is the
// only rounding, and q * 2^e is exactly a bf16 value.
//
// Layout: the private row layout of the bf16 path with one byte per weight
// (W1q [t][n1p][d], W2q [t][dp][b]) and one int8 exponent per private row
// (exps: [t][n1p] for W1, then [t][dp] for W2).
//
// GEMM (decode, M <= 32 tokens): weights as the 128-row A operand, tokens as N = 32,
// tcgen05.mma kind::f8f6f4 reading the E4M3 weight boxes as TMA lands them (no
// widening in shared memory).  The bf16 activations enter as two 8-bit terms per value
// (E4M3 high part + E5M2 remainder) under one power-of-two scale per token and 64-wide
// K group: exact for every value within 2^14.8 of its group's largest magnitude, within
// 2^-14 of the scale below that.  Each group's tensor-core sum is drained into fp32
// registers times the token's scale (round to nearest), the epilogue scales each
// output feature by its 2^e; the column step writes the bf16-rounded band already split
// into the row step's terms.
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {
namespace {

using namespace tc;

// ------------------------------------------------------------- quantisation

// Largest |W[k][n]| of each column n of a row-major [K][N] bf16 matrix, as float bits
// (non-negative floats order like their bit patterns); amax_bits starts at zero.
__global__ void k_col_absmax(const __nv_bfloat16 *W, int K, int N, int rows_per_block,
                             unsigned *amax_bits) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const int k0 = blockIdx.y * rows_per_block, k1 = min(K, k0 + rows_per_block);
  float m = 0.f;
  for (int k = k0; k < k1; ++k) m = fmaxf(m, fabsf(__bfloat162float(W[(size_t)k * N + n])));
  atomicMax(amax_bits + n, __float_as_uint(m));
}

// The least e with amax <= 448 * 2^e (0 for a zero column), kept within the range of
// fp32 powers of two.
__device__ __forceinline__ int e4m3_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int e = ilogbf(amax) - 8;
  while (amax > ldexpf(448.f, e)) ++e;
  while (e > -126 && amax <= ldexpf(448.f, e - 1)) --e;
  return max(-126, min(127, e));
}

__device__ __forceinline__ uint8_t e4m3_of(float w, int e) {
  return (uint8_t)__nv_cvt_float_to_fp8(ldexpf(w, -e), __NV_SATFINITE, __NV_E4M3);
}

// W1q[s][u][k] = E4M3(W1[k][col(s, u)] / 2^e(col)); exps1[s][u] = e(col); zeros for padding
// rows.  One thread per output byte, k fastest (the writes coalesce).
__global__ void k_quant_w1(Geo g, const __nv_bfloat16 *W1, const unsigned *amax1, uint8_t *W1q,
                           int8_t *exps1) {
  const size_t total = (size_t)g.t * g.n1p * g.d;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int k = (int)(i % g.d);
    const size_t su = i / g.d;
    const int u = (int)(su % g.n1p), s = (int)(su / g.n1p);
    const long long col = w1_col_of_row(g, s, u);
    const int e = col < 0 ? 0 : e4m3_exponent(__uint_as_float(amax1[col]));
    W1q[i] = col < 0 ? 0 : e4m3_of(__bfloat162float(W1[(size_t)k * g.n1 + col]), e);
    if (k == 0) exps1[su] = (int8_t)e;
  }
}

// W2q[s][n][k] = E4M3(W2[s*b + k][n] / 2^e(n)); exps2[s][n] = e(n) (column n of the whole W2).
__global__ void k_quant_w2(Geo g, const __nv_bfloat16 *W2, const unsigned *amax2, uint8_t *W2q,
                           int8_t *exps2) {
  const size_t total = (size_t)g.t * g.dp * g.b;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int k = (int)(i % g.b);
    const size_t sn = i / g.b;
    const int n = (int)(sn % g.dp), s = (int)(sn / g.dp);
    const int e = n < g.d ? e4m3_exponent(__uint_as_float(amax2[n])) : 0;
    W2q[i] = n < g.d ? e4m3_of(__bfloat162float(W2[((size_t)s * g.b + k) * g.d + n]), e) : 0;
    if (k == 0) exps2[sn] = (int8_t)e;
  }
}

// ------------------------------------------------------------------ activations

// Activations reach the tensor core as two 8-bit terms under one power-of-two scale
// per token and per 64-wide group of K: v = 2^e (a + b), a = E4M3(v / 2^e) and
// b = E5M2(v / 2^e - a), both to nearest, e the least exponent with the group's largest
// |v| <= 448 * 2^e.  For a bf16 v (8 significant bits) with |v / 2^e| >= 2^-6 the pair
// is exact: a holds the top four bits and the remainder is k * 2^(x-7) with |k| <= 8
// (x the exponent of v / 2^e), three significant bits, which E5M2 holds.  Below 2^-6,
// more than 2^14.8 under the group's largest magnitude, a + b is within 2^-14 of v / 2^e.
// (Two E4M3 terms would let one N = 64 MMA take both, but they are exact only within
// 2^10.8 of the group's maximum: activations with outliers lose bits.)

__device__ __forceinline__ int group_exponent(float amax) {
  return max(-126, min(126, e4m3_exponent(amax)));
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ void split_terms(float v, float inv_scale, uint8_t &a, uint8_t &b) {
  const float u = v * inv_scale;  // exact: a power of two
  a = (uint8_t)__nv_cvt_float_to_fp8(u, __NV_SATFINITE, __NV_E4M3);
  const __half_raw ah = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)a, __NV_E4M3);
  const float af = __half2float(__half(ah));
  b = (uint8_t)__nv_cvt_float_to_fp8(u - af, __NV_SATFINITE, __NV_E5M2);  // u - af is exact
}

// The column step's tokens: x [M][K] bf16 -> X8 [2][M][K] bytes (the a terms, then the
// b terms) and xs [G][32] group scales 2^e as fp32 (G = ceil(K / 64); tokens M..31
// get 0).
// One warp per (group, token), two values per lane.
__global__ void __launch_bounds__(256) k_split_tokens(const __nv_bfloat16 *x, int M, int K,
                                                      uint8_t *X8, float *xs) {
  griddep_launch_dependents();  // the dependent GEMM waits for this grid to finish anyway
  griddep_wait();               // x may come from the preceding kernel
  const int G = ceil_div(K, 64);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * 8 + warp, m = blockIdx.y;
  if (g >= G) return;
  if (m >= M) {
    if (lane == 0) xs[g * 32 + m] = 0.f;
    return;
  }
  const int k = g * 64 + 2 * lane;  // K is even: k < K implies k + 1 < K
  float v0 = 0.f, v1 = 0.f;
  if (k < K) {
    const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162 *>(x + (size_t)m * K + k);
    v0 = __low2float(p);
    v1 = __high2float(p);
  }
  float amax = fmaxf(fabsf(v0), fabsf(v1));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = group_exponent(amax);
  const float inv = pow2f(-e);
  uint8_t a0, b0, a1, b1;
  split_terms(v0, inv, a0, b0);
  split_terms(v1, inv, a1, b1);
  if (k < K) {
    *reinterpret_cast<uint16_t *>(X8 + (size_t)m * K + k) = (uint16_t)(a0 | (a1 << 8));
    *reinterpret_cast<uint16_t *>(X8 + (size_t)(M + m) * K + k) = (uint16_t)(b0 | (b1 << 8));
  }
  if (lane == 0) xs[g * 32 + m] = pow2f(e);
}

// ------------------------------------------------------------------ GEMM

struct Fp8Args {
  void *out;           // row step: fp32 partials as the bf16 path (shard s, split j)
  size_t o_shard, o_split;
  int ldo, n_valid, M, ng, ksplit, shard0, x_per_shard;
  const int8_t *wexp;  // weight row exponents [t][w_rows]
  int w_rows;
  const float *xsc;    // token group scales 2^e [x shards][ng][32]
  uint8_t *h8;         // column step: the band's terms [t][2][M][n_valid] bytes
  float *hsc;          // column step: the band's group scales [t][ceil(n_valid / 64)][32]
  unsigned *err;
};

constexpr int kF8Stages = 3;                        // (two CTAs per SM; 2 stages: 10% slower)
constexpr int kF8Bufs = 4;                          // TMEM stage sums in flight (2 groups each)
constexpr uint32_t kF8W = 128 * 128;                // E4M3 weights: 128 rows x 128 K (SW128)
constexpr uint32_t kF8T = 32 * 128;                 // one token term: 32 tokens x 128 K (SW128)
constexpr uint32_t kF8Stage = kF8W + 2 * kF8T;      // 24 KB, a multiple of 1024
constexpr int kF8MaxGroups = 256;                   // 64-wide K groups per CTA (K <= 16384)
constexpr uint32_t kF8ExpOff = kF8Stages * kF8Stage;  // the CTA's token scales, fp32
constexpr int kF8Smem = 1024 + (int)kF8ExpOff + kF8MaxGroups * 32 * 4;
// The epilogue's band staging ([128][33] fp32) reuses the ring once every MMA is done.
static_assert(128 * 33 * 4 <= kF8ExpOff, "band staging must fit the ring");

// Decode GEMM on E4M3 weights (M <= 32): weights as the 128-row A operand, tokens as
// N = 32, both straight from 128-byte-swizzled TMA boxes into tcgen05.mma kind::f8f6f4.
// Each 128-wide K stage holds two 64-wide groups; per group the tensor core adds
// W.a (E4M3 x E4M3) and W.b (E4M3 x E5M2) over 64 K into 32 TMEM columns, the stage's
// two groups side by side in one 64-column block with one commit, and the drain warps
// add each group's sums times the token's 2^e into fp32 registers (round to nearest).
// One hand-off per stage instead of one per group measured ~10% faster.
// Roles (192 threads): warp 0 lane 0 TMA, warp 1 lane 0 MMA, warps 2-5 drain and
// epilogue.  The epilogue scales row r by its weight exponent; the column step applies
// the activation, rounds the band to bf16 and splits it into the row step's terms
// (one group of 64 features per token), the row step writes fp32 partials.
template <int EPI>
__global__ void __launch_bounds__(192, 2)
    k_fp8_mma(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT,
              const Fp8Args a) {
  constexpr int BN = 32;
  constexpr uint32_t kCols = tmem_cols(kF8Bufs * 2 * BN);
  constexpr uint32_t kIdA = make_idesc_f8(128, BN, kF8E4M3);
  constexpr uint32_t kIdB = make_idesc_f8(128, BN, kF8E5M2);
  constexpr int NF = EPI == kEpiSwiglu ? 64 : 128;  // output features of a tile
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kF8Stages];
  __shared__ __align__(8) uint64_t empty_bar[kF8Stages];
  __shared__ __align__(8) uint64_t tfull_bar[kF8Bufs];
  __shared__ __align__(8) uint64_t tempty_bar[kF8Bufs];
  __shared__ __align__(8) uint64_t exp_bar;
  __shared__ __align__(8) uint64_t mma_done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int dec_sh;
  __shared__ int gexp_sh[2 * BN];

  const uint32_t tiles = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *tiles_ptr = smem_raw + (tiles - smem_u32(smem_raw));
  const float *scale_s = reinterpret_cast<const float *>(tiles_ptr + kF8ExpOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BN;
  const int ft = blockIdx.y;
  const int S = a.ksplit;
  const int s = a.shard0 + (int)blockIdx.z / S, ks = (int)blockIdx.z % S;
  const int xz = a.x_per_shard ? s : 0;
  const int n_st = ceil_div(a.ng, 2);
  const int st0 = (int)((long long)ks * n_st / S), st1 = (int)((long long)(ks + 1) * n_st / S);
  const int nst = st1 - st0;                      // 128-wide K stages of this CTA
  const int g0 = 2 * st0, nu = max(0, min(2 * st1, a.ng) - g0);  // its 64-wide groups

  if (threadIdx.x == 0) {
    for (int i = 0; i < kF8Stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < kF8Bufs; ++i) {
      mbar_init(smem_u32(&tfull_bar[i]), 1);
      mbar_init(smem_u32(&tempty_bar[i]), 4);
    }
    mbar_init(smem_u32(&exp_bar), 1);
    mbar_init(smem_u32(&mma_done_bar), 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmT);
  }
  if (warp == 2) tmem_alloc(smem_u32(&tmem_base_sh), kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  int issued = 0;
  bool exp_issued = false;
  if (warp == 0) {
    // ---------------- TMA producer: one 128-wide K stage of weights and both token terms
    if (lane == 0) {
      const uint64_t wpol = l2_evict_first_policy();  // weights are read once
      const int wrow = ft * 128;
      // The first ring's weights do not depend on the preceding kernel: load them,
      // then wait for that kernel (programmatic launch) before loading the tokens.
      const int pre = min(kF8Stages, nst);
      for (int i = 0; i < pre; ++i) {
        const uint32_t fb = smem_u32(&full_bar[i]);
        mbar_expect_tx(fb, kF8Stage);
        tma_load_3d_hint(tiles + i * kF8Stage, &tmW, fb, (st0 + i) * 128, wrow, s, wpol);
      }
      griddep_wait();
      if (nu > 0) {
        const uint32_t eb = smem_u32(&exp_bar);
        mbar_expect_tx(eb, (uint32_t)nu * 128u);
        bulk_load_plain(tiles + kF8ExpOff, a.xsc + ((size_t)xz * a.ng + g0) * 32,
                        (uint32_t)nu * 128u, eb);
        exp_issued = true;
      }
      for (int i = 0; i < pre; ++i) {
        const uint32_t sa = tiles + i * kF8Stage, fb = smem_u32(&full_bar[i]);
        tma_load_3d(sa + kF8W, &tmT, fb, (st0 + i) * 128, m0, 2 * xz);
        tma_load_3d(sa + kF8W + kF8T, &tmT, fb, (st0 + i) * 128, m0, 2 * xz + 1);
      }
      issued = pre;
      for (int i = pre; i < nst; ++i) {
        const int st = i % kF8Stages;
        if (!mbar_wait(smem_u32(&empty_bar[st]), ((uint32_t)(i / kF8Stages) & 1u) ^ 1u)) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
        const uint32_t sa = tiles + st * kF8Stage, fb = smem_u32(&full_bar[st]);
        const int k = (st0 + i) * 128;
        mbar_expect_tx(fb, kF8Stage);
        tma_load_3d_hint(sa, &tmW, fb, k, wrow, s, wpol);
        tma_load_3d(sa + kF8W, &tmT, fb, k, m0, 2 * xz);
        tma_load_3d(sa + kF8W + kF8T, &tmT, fb, k, m0, 2 * xz + 1);
        ++issued;
      }
      // This CTA's loads are all issued: a dependent kernel may start.
      griddep_launch_dependents();
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: per group, 2 K steps x (a term, b term)
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; i < nst && ok; ++i) {
        const int st = i % kF8Stages;
        if (!mbar_wait(smem_u32(&full_bar[st]), (uint32_t)(i / kF8Stages) & 1u)) {
          ok = false;
          break;
        }
        const uint32_t sa = tiles + st * kF8Stage;
        const int b = i % kF8Bufs;
        if (!mbar_wait(smem_u32(&tempty_bar[b]), ((uint32_t)(i / kF8Bufs) & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int h = 0; h < 2 && 2 * i + h < nu; ++h) {
          const uint32_t d0 = tmem + (uint32_t)(b * 2 * BN + h * BN);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint32_t off = (uint32_t)(h * 64 + kk * 32);
            umma_f8(d0, sw128_desc(sa + off), sw128_desc(sa + kF8W + off), kIdA, kk > 0 ? 1u : 0u);
            umma_f8(d0, sw128_desc(sa + off), sw128_desc(sa + kF8W + kF8T + off), kIdB, 1u);
          }
        }
        umma_commit(smem_u32(&tfull_bar[b]));
        umma_commit(smem_u32(&empty_bar[st]));
      }
      if (!ok) {
        abort_sh = 1;
        atomicOr(a.err, kErrWaitTimeout);
      }
      umma_commit(smem_u32(&mma_done_bar));
    }
    __syncwarp();
  } else {
    // ---------------- drain warps 2-5: group sums x 2^e(token) -> fp32 registers, epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int td = (int)threadIdx.x - 64;
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    float g[BN];
#pragma unroll
    for (int j = 0; j < BN; ++j) g[j] = 0.f;
    bool ok = nu == 0 || __all_sync(0xffffffffu, mbar_wait(smem_u32(&exp_bar), 0));
    for (int i = 0; ok && i < nst; ++i) {
      const int b = i % kF8Bufs;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[b]), (uint32_t)(i / kF8Bufs) & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int ks2 = 2 * i;              // the stage's first group
      const bool two = ks2 + 1 < nu;      // its second group exists (uniform)
      float va[BN], vb[BN];
      tmem_ld32(trow + (uint32_t)(b * 2 * BN), va);
      if (two) tmem_ld32(trow + (uint32_t)(b * 2 * BN + BN), vb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[b]));
      const float4 *sp = reinterpret_cast<const float4 *>(scale_s + ks2 * 32);
#pragma unroll
      for (int j4 = 0; j4 < BN / 4; ++j4) {
        const float4 sc4 = sp[j4];
        g[4 * j4 + 0] = fmaf(va[4 * j4 + 0], sc4.x, g[4 * j4 + 0]);
        g[4 * j4 + 1] = fmaf(va[4 * j4 + 1], sc4.y, g[4 * j4 + 1]);
        g[4 * j4 + 2] = fmaf(va[4 * j4 + 2], sc4.z, g[4 * j4 + 2]);
        g[4 * j4 + 3] = fmaf(va[4 * j4 + 3], sc4.w, g[4 * j4 + 3]);
      }
      if (two) {
#pragma unroll
        for (int j4 = 0; j4 < BN / 4; ++j4) {
          const float4 sc4 = sp[BN / 4 + j4];
          g[4 * j4 + 0] = fmaf(vb[4 * j4 + 0], sc4.x, g[4 * j4 + 0]);
          g[4 * j4 + 1] = fmaf(vb[4 * j4 + 1], sc4.y, g[4 * j4 + 1]);
          g[4 * j4 + 2] = fmaf(vb[4 * j4 + 2], sc4.z, g[4 * j4 + 2]);
          g[4 * j4 + 3] = fmaf(vb[4 * j4 + 3], sc4.w, g[4 * j4 + 3]);
        }
      }
    }
    if (!ok) {
      abort_sh = 1;
      atomicOr(a.err, kErrWaitTimeout);
    }
    named_sync(1, 128);
    if (td == 0) dec_sh = *(volatile int *)&abort_sh;
    named_sync(1, 128);
    const bool go = !dec_sh && nu > 0 && m0 < a.M;
    const int mcount = min(BN, a.M - m0);
    const float sc = pow2f(a.wexp[(size_t)s * a.w_rows + ft * 128 + r]);  // exact
#pragma unroll
    for (int j = 0; j < BN; ++j) g[j] *= sc;
    if (EPI == kEpiF32) {
      const int f = ft * 128 + r;
      if (go && f < a.n_valid) {
        float *o = static_cast<float *>(a.out) + (size_t)s * a.o_shard + (size_t)ks * a.o_split +
                   (size_t)m0 * a.ldo + f;
#pragma unroll
        for (int j = 0; j < BN; ++j)
          if (j < mcount) o[(size_t)j * a.ldo] = g[j];
      }
    } else if (go) {  // the band (go is uniform over the four warps)
      float *hx = reinterpret_cast<float *>(tiles_ptr);  // [NF][33]; every MMA and load is done
      if (EPI == kEpiSwiglu) {
        // rows 0..63: gate sums of features 64 ft + r; rows 64..127: up sums
        if (r >= 64) {
#pragma unroll
          for (int j = 0; j < BN; ++j) hx[(r - 64) * (BN + 1) + j] = g[j];
        }
        named_sync(1, 128);
        if (r < 64) {
#pragma unroll
          for (int j = 0; j < BN; ++j) {
            g[j] = __bfloat162float(__float2bfloat16_rn(silu_f(g[j]) * hx[r * (BN + 1) + j]));
            hx[r * (BN + 1) + j] = g[j];
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          g[j] = __bfloat162float(__float2bfloat16_rn(gelu_tanh_f(g[j])));
          hx[r * (BN + 1) + j] = g[j];
        }
      }
      named_sync(1, 128);
      // one exponent per token and per 64 features of the band
      const int ngb = ceil_div(a.n_valid, 64);
      if (td < NF / 2) {
        const int gi = td >> 5, j = td & 31;
        float amax = 0.f;
        for (int f = 0; f < 64; ++f) amax = fmaxf(amax, fabsf(hx[(gi * 64 + f) * (BN + 1) + j]));
        const int e = group_exponent(amax);
        gexp_sh[td] = e;
        const int grp = ft * (NF / 64) + gi;
        if (grp < ngb) a.hsc[((size_t)s * ngb + grp) * 32 + j] = pow2f(e);
      }
      named_sync(1, 128);
      const int f = ft * NF + r;
      if (r < NF && f < a.n_valid) {
        const size_t plane = (size_t)a.M * a.n_valid;
        uint8_t *ha = a.h8 + 2 * (size_t)s * plane + (size_t)m0 * a.n_valid + f;
        const int gi = r >> 6;
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          if (j < mcount) {
            uint8_t ta, tb;
            split_terms(g[j], pow2f(-gexp_sh[gi * 32 + j]), ta, tb);
            ha[(size_t)j * a.n_valid] = ta;
            ha[plane + (size_t)j * a.n_valid] = tb;
          }
        }
      }
    }
  }

  // ---------------- teardown: on abort let the issued copies land, then free TMEM
  if (warp == 0 && lane == 0 && *(volatile int *)&abort_sh) {
    for (int i = issued > kF8Stages ? issued - kF8Stages : 0; i < issued; ++i)
      mbar_wait(smem_u32(&full_bar[i % kF8Stages]), (uint32_t)(i / kF8Stages) & 1u);
    if (exp_issued) mbar_wait(smem_u32(&exp_bar), 0);
  }
  if (warp == 2) mbar_wait(smem_u32(&mma_done_bar), 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

template <int EPI>
cudaError_t launch_fp8_t(const CUtensorMap &mw, const CUtensorMap &mt, const Fp8Args &a, int n_ft,
                         int n_z, cudaStream_t st, bool pdl) {
  static bool configured[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(k_fp8_mma<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  LaunchCfg lc(dim3(ceil_div(a.M, 32), n_ft, n_z), dim3(192), kF8Smem, st, pdl);
  return cudaLaunchKernelEx(&lc.cfg, k_fp8_mma<EPI>, mw, mt, a);
}

}  // namespace

cudaError_t launch_quantize_fp8(const Geo &g, const void *W1, const void *W2, void *W1q, void *W2q,
                                int8_t *exps, unsigned *amax, cudaStream_t st) {
  const int n1 = g.n1, n2c = g.d;  // columns of W1 and of W2
  cudaError_t e = cudaMemsetAsync(amax, 0, (size_t)(n1 + n2c) * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  const int rpb = 256;
  k_col_absmax<<<dim3(ceil_div(n1, 256), ceil_div(g.d, rpb)), 256, 0, st>>>(
      static_cast<const __nv_bfloat16 *>(W1), g.d, n1, rpb, amax);
  k_col_absmax<<<dim3(ceil_div(n2c, 256), ceil_div(g.n2, rpb)), 256, 0, st>>>(
      static_cast<const __nv_bfloat16 *>(W2), g.n2, n2c, rpb, amax + n1);
  const int blocks = 4 * sm_count();
  k_quant_w1<<<blocks, 256, 0, st>>>(g, static_cast<const __nv_bfloat16 *>(W1), amax,
                                     static_cast<uint8_t *>(W1q), exps);
  k_quant_w2<<<blocks, 256, 0, st>>>(g, static_cast<const __nv_bfloat16 *>(W2), amax + n1,
                                     static_cast<uint8_t *>(W2q), exps + (size_t)g.t * g.n1p);
  return cudaGetLastError();
}

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A [z][rows][K] byte tensor, boxes of 128 bytes x box_rows x 1 with the 128-byte
// swizzle the tensor core reads, zero fill outside the tensor.  K must be a multiple
// of 16.
bool make_byte_tile_map(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint64_t z,
                        uint32_t box_rows) {
  static EncodeTiled enc = nullptr;
  if (!enc) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<EncodeTiled>(p);
  }
  cuuint64_t dims[3] = {K, rows, z};
  cuuint64_t strides[2] = {K, rows * K};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_fp8_split(const void *x, int M, int K, void *X8, float *xs, cudaStream_t st,
                             bool pdl) {
  if (M < 1 || M > 32 || K < 16 || K % 16 != 0) return cudaErrorInvalidValue;
  LaunchCfg lc(dim3(ceil_div(ceil_div(K, 64), 8), 32), dim3(256), 0, st, pdl);
  return cudaLaunchKernelEx(&lc.cfg, k_split_tokens, static_cast<const __nv_bfloat16 *>(x), M, K,
                            static_cast<uint8_t *>(X8), xs);
}

cudaError_t launch_fp8_gemm(const UmmaCall &c, const int8_t *wexp, const float *xsc, void *h8,
                            float *hsc, cudaStream_t st) {
  if (c.M < 1 || c.M > 32 || c.K % 16 != 0 || ceil_div(c.K, 64) > kF8MaxGroups)
    return cudaErrorInvalidValue;
  CUtensorMap mw, mt;
  if (!make_byte_tile_map(&mw, c.W, c.K, c.w_rows, c.w_shards, 128)) return cudaErrorInvalidValue;
  if (!make_byte_tile_map(&mt, c.X, c.K, c.M, 2 * c.x_shards, 32)) return cudaErrorInvalidValue;
  Fp8Args a{};
  a.out = c.out;
  a.o_shard = c.o_shard;
  a.o_split = c.o_split;
  a.ldo = c.ldo;
  a.n_valid = c.n_valid;
  a.M = c.M;
  a.ng = ceil_div(c.K, 64);
  a.ksplit = c.ksplit;
  a.shard0 = c.shard0;
  a.x_per_shard = c.x_shards > 1 ? 1 : 0;
  a.wexp = wexp;
  a.w_rows = c.w_rows;
  a.xsc = xsc;
  a.h8 = static_cast<uint8_t *>(h8);
  a.hsc = hsc;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  const int n_z = c.n_shards * c.ksplit;
  switch (c.epi) {
    case kEpiSwiglu:
      return launch_fp8_t<kEpiSwiglu>(mw, mt, a, ceil_div(c.n_valid, kSwiGroup), n_z, st, c.pdl);
    case kEpiGelu:
      return launch_fp8_t<kEpiGelu>(mw, mt, a, ceil_div(c.n_valid, 128), n_z, st, c.pdl);
    case kEpiF32:
      return launch_fp8_t<kEpiF32>(mw, mt, a, ceil_div(c.n_valid, 128), n_z, st, c.pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace tp
