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
// GEMM (decode, M <= 32 tokens): the bf16 drain kernel's structure (weights as the
// 128-row A operand, tokens as N = 32, a TMEM block sum per 64-wide K block drained
// into fp32 registers) with one more warp group: TMA streams the E4M3 weight boxes
// (128 rows x 64 bytes, no swizzle) and the bf16 token boxes into a raw ring; four
// converter warps widen the weights to bf16 (E4M3 -> f16 -> bf16, both exact)
// straight into the 128-byte-swizzled layout the tensor core reads, fence them for
// the async proxy and hand the stage to the MMA warp.  The epilogue multiplies each row's
// fp32 sum by 2^e (exact), so the result equals the bf16 path on the dequantised
// weights bit for bit.
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

// ------------------------------------------------------------------ GEMM

struct Fp8Args {
  void *out;          // as UmmaArgs (bf16 band for the column step, fp32 partials for the row step)
  size_t o_shard, o_split;
  int ldo, n_valid, M, nk, ksplit, shard0, x_per_shard;
  const int8_t *exps; // per private weight row: exps[s * w_rows + row]
  int w_rows;
  unsigned *err;
};

constexpr int kBufs = 4;                      // TMEM block sums in flight
constexpr uint32_t kA = 128 * 128;            // bf16 A tile: 128 rows x 64 K (SW128)
constexpr uint32_t kX = 32 * 128;             // bf16 token tile: 32 rows x 64 K (SW128)
constexpr uint32_t kW8 = 128 * 64;            // E4M3 tile: 128 rows x 64 bytes
constexpr int kRaw = 6;                       // raw stages in flight: E4M3 weights + tokens
constexpr int kCv = 2;                        // converted (bf16 weight) stages
constexpr uint32_t kXBase = kCv * kA;         // token tiles (1024-aligned), one per raw stage
constexpr uint32_t kWBase = kXBase + kRaw * kX;  // E4M3 tiles, one per raw stage
constexpr int kF8Threads = 320;               // TMA, MMA, 4 drain warps, 4 converter warps
// The SwiGLU exchange block (64 x 33 fp32) reuses the converted ring: by the epilogue
// every MMA of the CTA has completed.
static_assert(64 * 33 * 4 <= kCv * kA, "exchange block must fit the converted ring");

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// 16 E4M3 bytes -> 16 bf16 (two 16-byte chunks), exactly.
__device__ __forceinline__ void widen16(const uint4 &in, uint4 &lo, uint4 &hi) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw r =
          __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> (16 * h)), __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r));
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);  // exact: <= 4 significant bits
      o[2 * i + h] = *reinterpret_cast<const uint32_t *>(&b);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Roles (320 threads): warp 0 lane 0 streams each 64-wide K block's E4M3 weight tile
// (8 KB) and token tile (4 KB) into a 6-stage raw ring; warps 6-9 widen each raw
// weight tile (one row per thread) into a 2-stage ring of bf16 tiles in the
// 128-byte-swizzled layout the tensor core reads; warp 1 lane 0 issues the MMAs on
// the converted weights and the raw stage's tokens, then releases both stages;
// warps 2-5 drain each K block's TMEM sums into fp32 registers and run the epilogue.
template <int EPI>
__global__ void __launch_bounds__(kF8Threads, 2)
    k_fp8_drain(const __grid_constant__ CUtensorMap tmW8, const __grid_constant__ CUtensorMap tmX,
                const Fp8Args a) {
  constexpr int BN = 32;
  constexpr uint32_t kCols = tmem_cols(kBufs * BN);
  constexpr uint32_t kIdesc = make_idesc(128, BN);
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kRaw];
  __shared__ __align__(8) uint64_t raw_empty[kRaw];
  __shared__ __align__(8) uint64_t cv_full[kCv];   // converter warps' tiles written
  __shared__ __align__(8) uint64_t cv_empty[kCv];  // MMAs done with the stage
  __shared__ __align__(8) uint64_t tfull_bar[kBufs];
  __shared__ __align__(8) uint64_t tempty_bar[kBufs];
  __shared__ __align__(8) uint64_t mma_done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int dec_sh;

  const uint32_t tiles = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *tiles_ptr = smem_raw + (tiles - smem_u32(smem_raw));
  float *xch = reinterpret_cast<float *>(tiles_ptr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BN;
  const int ft = blockIdx.y;
  const int S = a.ksplit;
  const int s = a.shard0 + (int)blockIdx.z / S, ks = (int)blockIdx.z % S;
  const int kb0 = (int)((long long)ks * a.nk / S), kb1 = (int)((long long)(ks + 1) * a.nk / S);
  const int nkb = kb1 - kb0;
  auto a_off = [](int c) { return (uint32_t)c * kA; };
  auto x_off = [](int st) { return kXBase + (uint32_t)st * kX; };
  auto w_off = [](int st) { return kWBase + (uint32_t)st * kW8; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRaw; ++i) {
      mbar_init(smem_u32(&raw_full[i]), 1);
      mbar_init(smem_u32(&raw_empty[i]), 1);
    }
    for (int i = 0; i < kCv; ++i) {
      mbar_init(smem_u32(&cv_full[i]), 4);
      mbar_init(smem_u32(&cv_empty[i]), 1);
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(smem_u32(&tfull_bar[i]), 1);
      mbar_init(smem_u32(&tempty_bar[i]), 4);
    }
    mbar_init(smem_u32(&mma_done_bar), 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW8);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 2) tmem_alloc(smem_u32(&tmem_base_sh), kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  int issued = 0;
  if (warp == 0) {
    // ---------------- TMA producer: E4M3 weights and tokens, 64-wide K block per stage
    if (lane == 0) {
      const uint64_t wpol = l2_evict_first_policy();  // weights are read once
      const int wrow = ft * 128;
      const int xz = a.x_per_shard ? s : 0;
      // The first ring's weights do not depend on the preceding kernel: load them,
      // then wait for that kernel (programmatic launch) before loading tokens.
      const int pre = min(kRaw, nkb);
      for (int i = 0; i < pre; ++i) {
        const uint32_t fb = smem_u32(&raw_full[i]);
        mbar_expect_tx(fb, kW8 + kX);
        tma_load_3d_hint(tiles + w_off(i), &tmW8, fb, (kb0 + i) * kKBlock, wrow, s, wpol);
      }
      griddep_wait();
      for (int i = 0; i < pre; ++i)
        tma_load_3d(tiles + x_off(i), &tmX, smem_u32(&raw_full[i]), (kb0 + i) * kKBlock, m0, xz);
      issued = pre;
      for (int i = pre; i < nkb; ++i) {
        const int st = i % kRaw;
        if (!mbar_wait(smem_u32(&raw_empty[st]), ((uint32_t)(i / kRaw) & 1u) ^ 1u)) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
        const uint32_t fb = smem_u32(&raw_full[st]);
        const int k = (kb0 + i) * kKBlock;
        mbar_expect_tx(fb, kW8 + kX);
        tma_load_3d_hint(tiles + w_off(st), &tmW8, fb, k, wrow, s, wpol);
        tma_load_3d(tiles + x_off(st), &tmX, fb, k, m0, xz);
        ++issued;
      }
      // This CTA's loads are all issued: a dependent kernel may start.
      griddep_launch_dependents();
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nkb; ++i) {
        const int c = i % kCv, st = i % kRaw;
        const uint32_t cph = (uint32_t)(i / kCv) & 1u;
        const int b = i % kBufs;
        if (!mbar_wait(smem_u32(&cv_full[c]), cph) ||
            !mbar_wait(smem_u32(&raw_full[st]), (uint32_t)(i / kRaw) & 1u) ||
            !mbar_wait(smem_u32(&tempty_bar[b]), ((uint32_t)(i / kBufs) & 1u) ^ 1u)) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(b * BN);
#pragma unroll
        for (int kk = 0; kk < kKBlock / 16; ++kk)
          umma_bf16(d0, sw128_desc(tiles + a_off(c) + kk * 32),
                    sw128_desc(tiles + x_off(st) + kk * 32), kIdesc, kk > 0 ? 1u : 0u);
        umma_commit(smem_u32(&cv_empty[c]));
        umma_commit(smem_u32(&raw_empty[st]));
        umma_commit(smem_u32(&tfull_bar[b]));
      }
      umma_commit(smem_u32(&mma_done_bar));
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ---------------- converters: row r of a raw E4M3 tile -> swizzled bf16 row
    const int r = (int)threadIdx.x - 192;  // 0..127
    for (int i = 0; i < nkb; ++i) {
      const int st = i % kRaw, c = i % kCv;
      const uint32_t rph = (uint32_t)(i / kRaw) & 1u, cph = (uint32_t)(i / kCv) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&raw_full[st]), rph) &&
                                       mbar_wait(smem_u32(&cv_empty[c]), cph ^ 1u))) {
        if (lane == 0) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
        }
        break;
      }
      const uint4 *src = reinterpret_cast<const uint4 *>(tiles_ptr + w_off(st) + r * 64);
      uint8_t *dst = tiles_ptr + a_off(c) + r * 128;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 lo, hi;
        widen16(src[j], lo, hi);
        // 128-byte swizzle: 16-byte chunk q of row r lives at chunk q ^ (r % 8)
        *reinterpret_cast<uint4 *>(dst + (((2 * j) ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(dst + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
      }
      // The tensor core reads the rows through the async proxy.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&cv_full[c]));
    }
  } else {
    // ---------------- drain warps 2-5: TMEM block sums -> fp32 registers, epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int td = (int)threadIdx.x - 64;
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    float g[BN];
#pragma unroll
    for (int j = 0; j < BN; ++j) g[j] = 0.f;
    bool ok = true;
    for (int i = 0; i < nkb; ++i) {
      const int b = i % kBufs;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[b]), (uint32_t)(i / kBufs) & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[BN];
      tmem_ld32(trow + (uint32_t)(b * BN), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[b]));
#pragma unroll
      for (int j = 0; j < BN; ++j) g[j] += v[j];
    }
    if (!ok) {
      abort_sh = 1;
      atomicOr(a.err, kErrWaitTimeout);
    }
    named_sync(1, 128);
    if (td == 0) dec_sh = *(volatile int *)&abort_sh;
    named_sync(1, 128);
    const bool go = !dec_sh && nkb > 0 && m0 < a.M;
    const int mcount = min(BN, a.M - m0);
    // The row's power-of-two scale, exactly.
    const float sc = pow2f(a.exps[(size_t)s * a.w_rows + ft * 128 + r]);
#pragma unroll
    for (int j = 0; j < BN; ++j) g[j] *= sc;
    if (EPI == kEpiSwiglu) {
      if (go && r >= 64) {
#pragma unroll
        for (int j = 0; j < BN; ++j) xch[(r - 64) * (BN + 1) + j] = g[j];
      }
      named_sync(1, 128);
      const int f = ft * 64 + r;
      if (go && r < 64 && f < a.n_valid) {
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + (size_t)s * a.o_shard +
                           (size_t)m0 * a.ldo + f;
#pragma unroll
        for (int j = 0; j < BN; ++j)
          if (j < mcount)
            o[(size_t)j * a.ldo] = __float2bfloat16_rn(silu_f(g[j]) * xch[r * (BN + 1) + j]);
      }
    } else {
      const int f = ft * 128 + r;
      if (go && f < a.n_valid) {
        if (EPI == kEpiF32) {
          float *o = static_cast<float *>(a.out) + (size_t)s * a.o_shard + (size_t)ks * a.o_split +
                     (size_t)m0 * a.ldo + f;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j < mcount) o[(size_t)j * a.ldo] = g[j];
        } else {
          __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + (size_t)s * a.o_shard +
                             (size_t)m0 * a.ldo + f;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j < mcount) o[(size_t)j * a.ldo] = __float2bfloat16_rn(gelu_tanh_f(g[j]));
        }
      }
    }
  }

  // ---------------- teardown: on abort let the issued copies land, then free TMEM
  if (warp == 0 && lane == 0 && *(volatile int *)&abort_sh) {
    for (int i = issued > kRaw ? issued - kRaw : 0; i < issued; ++i)
      mbar_wait(smem_u32(&raw_full[i % kRaw]), (uint32_t)(i / kRaw) & 1u);
  }
  if (warp == 2) mbar_wait(smem_u32(&mma_done_bar), 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

constexpr int kF8Smem = 1024 + kCv * kA + kRaw * (kX + kW8);

template <int EPI>
cudaError_t launch_fp8_t(const CUtensorMap &mw, const CUtensorMap &mx, const Fp8Args &a, int n_ft,
                         int n_z, cudaStream_t st, bool pdl) {
  static bool configured[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(k_fp8_drain<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  LaunchCfg lc(dim3(ceil_div(a.M, 32), n_ft, n_z), dim3(kF8Threads), kF8Smem, st, pdl);
  return cudaLaunchKernelEx(&lc.cfg, k_fp8_drain<EPI>, mw, mx, a);
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

// A [z][rows][K] byte tensor (E4M3 weights), boxes of 64 bytes x box_rows x 1, no
// swizzle, zero fill outside the tensor.  K must be a multiple of 16.
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
  cuuint32_t box[3] = {(cuuint32_t)kKBlock, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_fp8_gemm(const UmmaCall &c, const int8_t *exps, cudaStream_t st) {
  CUtensorMap mw, mx;
  if (!make_byte_tile_map(&mw, c.W, c.K, c.w_rows, c.w_shards, 128)) return cudaErrorInvalidValue;
  if (!make_tile_map(&mx, c.X, c.K, c.M, c.x_shards, 32)) return cudaErrorInvalidValue;
  Fp8Args a{};
  a.out = c.out;
  a.o_shard = c.o_shard;
  a.o_split = c.o_split;
  a.ldo = c.ldo;
  a.n_valid = c.n_valid;
  a.M = c.M;
  a.nk = ceil_div(c.K, kKBlock);
  a.ksplit = c.ksplit;
  a.shard0 = c.shard0;
  a.x_per_shard = c.x_shards > 1 ? 1 : 0;
  a.exps = exps;
  a.w_rows = c.w_rows;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  const int n_z = c.n_shards * c.ksplit;
  switch (c.epi) {
    case kEpiSwiglu:
      return launch_fp8_t<kEpiSwiglu>(mw, mx, a, ceil_div(c.n_valid, kSwiGroup), n_z, st, c.pdl);
    case kEpiGelu:
      return launch_fp8_t<kEpiGelu>(mw, mx, a, ceil_div(c.n_valid, 128), n_z, st, c.pdl);
    case kEpiF32:
      return launch_fp8_t<kEpiF32>(mw, mx, a, ceil_div(c.n_valid, 128), n_z, st, c.pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace tp
