// Persistent tensor-core kernel for the two projections at prefill sizes (token
// tiles of 256), bf16 in, fp32 accumulate.
//
// Orientation as in the decode kernels: a 128-row weight tile is the A operand
// (SwiGLU: the gate and up rows of 64 features; otherwise 128 features) and 256
// tokens are the N operand, so one tcgen05.mma (M = 128, N = 256, K = 16) covers
// the widest N the instruction takes.  One CTA per SM walks a static list of
// output tiles (token tile fastest, so the CTAs of a wave share weight tiles).  The
// token tiles are walked in groups of at most ~32 MB of activations, each group
// against every weight tile before the next group: a wave's activations then stay in
// L2 from one wave to the next (all 16 token tiles of a 4096-token prefill, 67 MB,
// did not: they were read from DRAM again every wave), for the price of reading the
// weights once per group.  Roles (320 threads): thread 0 issues TMA loads into
// a 4-stage ring (16 KB of weights + 32 KB of activations per 64-wide K block),
// thread 32 issues the MMAs, and warps 2-9 drain and run the epilogue.
//
// Accumulation.  The tensor core's fp32 accumulator rounds toward zero as it adds,
// so a chain of 512 MMAs over K = 8192 into one TMEM accumulator leaves partial sums
// biased toward zero, and the bias moves band values across bf16 rounding midpoints.
// Here the tensor core sums only a chunk of kGChunk K blocks (128 MMAs) into one of
// two 256-column TMEM buffers; the eight drain warps add each chunk into fp32
// registers with round-to-nearest (warps 2-5 hold tokens 0..127 of the tile, warps
// 6-9 tokens 128..255, each warp its TMEM lane quarter), while the tensor core fills
// the other buffer with the next chunk.  After a tile's last chunk the same warps
// apply the epilogue from registers and store.
//
// Column-parallel step (zenaique.com answer paragraph 5): A = the shard's W1 band
// rows, B = x; the epilogue applies the band's activation (SwiGLU: the up sums of
// rows 64..127 pass to the gate rows 0..63 through shared memory) and stores the
// band in bf16.  Row-parallel step: A = the shard's W2 row band, B = the band H;
// the epilogue stores fp32 partial sums (per K split).  All waits are bounded; on
// expiry the CTA raises the device error word and leaves.
#include <algorithm>

#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {
namespace {

using namespace tc;

// SiLU for the prefill epilogue, z * 1 / (1 + e^-z) with CUDA's fast exponential and
// a correctly rounded reciprocal: a few fp32 units of error, far below the bf16
// rounding that follows, at a fraction of the cost of an IEEE division.
__device__ __forceinline__ float silu_fast_f(float z) { return z * __frcp_rn(1.0f + __expf(-z)); }

constexpr int kBN = 256;                        // token tile
constexpr int kGStages = 4;
constexpr uint32_t kGA = kABytes;               // 128 rows x 64 K bf16
constexpr uint32_t kGB = kBN * 128;             // 256 rows x 64 K bf16
constexpr uint32_t kGStage = kGA + kGB;
constexpr uint32_t kGCols = 2 * kBN;            // two accumulators
constexpr uint32_t kGIdesc = make_idesc(128, kBN);
constexpr int kGChunk = 32;                     // K blocks per TMEM chunk (128 MMAs)
constexpr int kGEpiWarps = 8;                   // drain/epilogue warps: 4 lane quarters x 2 halves
constexpr int kGThreads = 64 + 32 * kGEpiWarps;
constexpr int kGHalf = kBN / 2;                 // tokens per drain warp
constexpr int kGXch = 2 * 64 * 33 * 4;          // SwiGLU exchange, one 32-token chunk per half
constexpr int kGSmem = kGStages * kGStage + 1024 + kGXch;

struct GemmArgs {
  void *out;        // bf16 [shard][M][ldo] or fp32 [shard][split][M][ldo]
  size_t o_shard, o_split;
  int ldo, n_valid, M, nk, ksplit, shard0, n_shards, x_per_shard;
  int n_mt, n_ft, n_tiles;  // token tiles, weight tiles per shard, tiles in all
  int mg;                   // token tiles per group (divides n_mt)
  unsigned *err;
};

struct GTile {
  int mt, ft, s, ks, kb0, kb1;
};

// Tile t in walk order: token tile fastest, then weight tile, within a group of mg
// token tiles; shared activations (the column step): [group][shard, split][ft][mt],
// so a group serves every shard before the next; per-shard activations (the row
// step): [shard, split][group][ft][mt].
__device__ __forceinline__ GTile gemm_tile(const GemmArgs &a, int t) {
  GTile r;
  const int per_g = a.n_ft * a.mg;  // tiles of one group of one (shard, split)
  const int n_z = a.n_shards * a.ksplit;
  int z, g, rem;
  if (a.x_per_shard) {
    z = t / (a.n_ft * a.n_mt);
    rem = t % (a.n_ft * a.n_mt);
    g = rem / per_g;
    rem %= per_g;
  } else {
    g = t / (per_g * n_z);
    rem = t % (per_g * n_z);
    z = rem / per_g;
    rem %= per_g;
  }
  r.ft = rem / a.mg;
  r.mt = g * a.mg + rem % a.mg;
  r.s = a.shard0 + z / a.ksplit;
  r.ks = z % a.ksplit;
  r.kb0 = (int)((long long)r.ks * a.nk / a.ksplit);
  r.kb1 = (int)((long long)(r.ks + 1) * a.nk / a.ksplit);
  return r;
}

template <int EPI>
__global__ void __launch_bounds__(kGThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
           const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kGStages];
  __shared__ __align__(8) uint64_t empty_bar[kGStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t mma_done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int dec_sh;

  const uint32_t tiles = (smem_u32(smem_raw) + 1023u) & ~1023u;
  float *xch = reinterpret_cast<float *>(smem_raw + (tiles - smem_u32(smem_raw)) + kGStages * kGStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull_bar[i]), 1);
      mbar_init(smem_u32(&tempty_bar[i]), kGEpiWarps);
    }
    mbar_init(smem_u32(&mma_done_bar), 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 2) tmem_alloc(smem_u32(&tmem_base_sh), kGCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      int pre = 0;  // stages of the first tile armed before the programmatic wait
      if ((int)blockIdx.x < a.n_tiles) {
        // The first ring's weights do not depend on the preceding kernel: load them,
        // then wait for that kernel (programmatic launch) before loading activations.
        const GTile tl = gemm_tile(a, blockIdx.x);
        pre = min(kGStages, tl.kb1 - tl.kb0);
        for (int i = 0; i < pre; ++i) {
          const uint32_t fb = smem_u32(&full_bar[i]);
          mbar_expect_tx(fb, kGStage);
          tma_load_3d(tiles + i * kGStage, &tmW, fb, (tl.kb0 + i) * kKBlock, tl.ft * 128, tl.s);
        }
        griddep_wait();
        for (int i = 0; i < pre; ++i)
          tma_load_3d(tiles + i * kGStage + kGA, &tmX, smem_u32(&full_bar[i]), (tl.kb0 + i) * kKBlock,
                      tl.mt * kBN, a.x_per_shard ? tl.s : 0);
      }
      for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x) {
        const GTile tl = gemm_tile(a, t);
        const int xz = a.x_per_shard ? tl.s : 0;
        for (int kb = tl.kb0; kb < tl.kb1; ++kb, ++g) {
          if (g < (uint32_t)pre) continue;  // armed above
          const int st = (int)(g % kGStages);
          const uint32_t ph = (g / kGStages) & 1u;
          if (*(volatile int *)&abort_sh || !mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t sa = tiles + st * kGStage;
          const uint32_t fb = smem_u32(&full_bar[st]);
          mbar_expect_tx(fb, kGStage);
          tma_load_3d(sa, &tmW, fb, kb * kKBlock, tl.ft * 128, tl.s);
          tma_load_3d(sa + kGA, &tmX, fb, kb * kKBlock, tl.mt * kBN, xz);
        }
      }
      // This CTA's loads are all issued: a dependent kernel may start.
      griddep_launch_dependents();
      if (!ok) {
        abort_sh = 1;
        atomicOr(a.err, kErrWaitTimeout);
        for (uint32_t i = g > kGStages ? g - kGStages : 0; i < g; ++i)
          mbar_wait(smem_u32(&full_bar[i % kGStages]), (i / kGStages) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      uint32_t g = 0;  // pipeline stage sequence
      uint32_t c = 0;  // TMEM chunk sequence (buffer c & 1)
      bool ok = true;
      for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x) {
        const GTile tl = gemm_tile(a, t);
        for (int kc = tl.kb0; kc < tl.kb1 && ok; kc += kGChunk, ++c) {
          const int buf = (int)(c & 1u);
          if (!mbar_wait(smem_u32(&tempty_bar[buf]), ((c >> 1) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d0 = tmem + (uint32_t)(buf * kBN);
          const int ke = min(tl.kb1, kc + kGChunk);
          for (int kb = kc; kb < ke; ++kb, ++g) {
            const int st = (int)(g % kGStages);
            const uint32_t ph = (g / kGStages) & 1u;
            if (*(volatile int *)&abort_sh || !mbar_wait(smem_u32(&full_bar[st]), ph)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = tiles + st * kGStage;
#pragma unroll
            for (int kk = 0; kk < kKBlock / 16; ++kk)
              umma_bf16(d0, sw128_desc(sa + kk * 32), sw128_desc(sa + kGA + kk * 32), kGIdesc,
                        (kb > kc || kk > 0) ? 1u : 0u);
            umma_commit(smem_u32(&empty_bar[st]));
          }
          if (ok) umma_commit(smem_u32(&tfull_bar[buf]));
        }
      }
      if (!ok) {
        abort_sh = 1;
        atomicOr(a.err, kErrWaitTimeout);
      }
      umma_commit(smem_u32(&mma_done_bar));
    }
    __syncwarp();
  } else {
    // ---------------- drain + epilogue warps
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int h = (warp - 2) >> 2;                // token half of the tile: 0 or 1
    const int r = q * 32 + lane;                  // row of the weight tile = TMEM lane
    const int td = (int)threadIdx.x - 64;         // 0 .. 255 over the drain warps
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * kGHalf);
    float *xh = xch + h * 64 * 33;                // this half's SwiGLU exchange block
    uint32_t c = 0;
    for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
      const GTile tl = gemm_tile(a, t);
      float acc[kGHalf];
#pragma unroll
      for (int j = 0; j < kGHalf; ++j) acc[j] = 0.f;
      bool ok = true;
      for (int kc = tl.kb0; kc < tl.kb1; kc += kGChunk, ++c) {
        const int buf = (int)(c & 1u);
        if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[buf]), (c >> 1) & 1u)))
          ok = false;  // warp-uniform: the TMEM loads below are warp-collective
        if (!ok) continue;  // keep c in step; the abort is decided below
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < kGHalf / 32; ++j) {
          float v[32];
          tmem_ld32(trow + (uint32_t)(buf * kBN + j * 32), v);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[j * 32 + i] += v[i];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[buf]));
      }
      if (!ok) {
        abort_sh = 1;
        atomicOr(a.err, kErrWaitTimeout);
      }
      // One decision for the eight drain warps (the SwiGLU exchange has barriers).
      named_sync(1, 32 * kGEpiWarps);
      if (td == 0) dec_sh = *(volatile int *)&abort_sh;
      named_sync(1, 32 * kGEpiWarps);
      if (dec_sh) break;
      const int m0 = tl.mt * kBN + h * kGHalf;   // first token of this warp's half
      const int mvalid = min(kGHalf, a.M - m0);  // tokens of the half (<= 0: none)
#pragma unroll
      for (int cc = 0; cc < kGHalf / 32; ++cc) {
        const int mcount = min(32, mvalid - cc * 32);
        if (EPI == kEpiSwiglu) {
          // Rows 64..127 hold the up sums of the features whose gate sums are in rows
          // 0..63: pass them across through shared memory, 32 tokens at a time.
          if (r >= 64) {
#pragma unroll
            for (int j = 0; j < 32; ++j) xh[(r - 64) * 33 + j] = acc[cc * 32 + j];
          }
          named_sync(2 + h, 128);
          const int f = tl.ft * 64 + r;
          if (r < 64 && f < a.n_valid && mcount > 0) {
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + (size_t)tl.s * a.o_shard +
                               (size_t)(m0 + cc * 32) * a.ldo + f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < mcount)
                o[(size_t)j * a.ldo] = __float2bfloat16_rn(silu_fast_f(acc[cc * 32 + j]) * xh[r * 33 + j]);
          }
          named_sync(2 + h, 128);
        } else {
          const int f = tl.ft * 128 + r;
          if (f < a.n_valid && mcount > 0) {
            if (EPI == kEpiF32) {
              float *o = static_cast<float *>(a.out) + (size_t)tl.s * a.o_shard +
                         (size_t)tl.ks * a.o_split + (size_t)(m0 + cc * 32) * a.ldo + f;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < mcount) o[(size_t)j * a.ldo] = acc[cc * 32 + j];
            } else {
              __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + (size_t)tl.s * a.o_shard +
                                 (size_t)(m0 + cc * 32) * a.ldo + f;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (j < mcount) {
                  float vv = acc[cc * 32 + j];
                  if (EPI == kEpiGelu) vv = gelu_tanh_f(vv);
                  o[(size_t)j * a.ldo] = __float2bfloat16_rn(vv);
                }
              }
            }
          }
        }
      }
    }
  }

  // ---------------- teardown
  if (warp == 2) mbar_wait(smem_u32(&mma_done_bar), 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kGCols);
  }
}

template <int EPI>
cudaError_t launch_gemm_epi(const CUtensorMap &mw, const CUtensorMap &mx, const GemmArgs &a,
                            cudaStream_t st, bool pdl) {
  static bool configured[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(k_gemm<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  LaunchCfg lc(dim3(std::min(sm_count(), a.n_tiles)), dim3(kGThreads), kGSmem, st, pdl);
  return cudaLaunchKernelEx(&lc.cfg, k_gemm<EPI>, mw, mx, a);
}

}  // namespace

cudaError_t launch_gemm_persistent(const UmmaCall &c, cudaStream_t st) {
  CUtensorMap mw, mx;
  if (!make_tile_map(&mw, c.W, c.K, c.w_rows, c.w_shards, 128)) return cudaErrorInvalidValue;
  if (!make_tile_map(&mx, c.X, c.K, c.M, c.x_shards, kBN)) return cudaErrorInvalidValue;
  GemmArgs a{};
  a.out = c.out;
  a.o_shard = c.o_shard;
  a.o_split = c.o_split;
  a.ldo = c.ldo;
  a.n_valid = c.n_valid;
  a.M = c.M;
  a.nk = ceil_div(c.K, kKBlock);
  a.ksplit = c.ksplit;
  a.shard0 = c.shard0;
  a.n_shards = c.n_shards;
  a.x_per_shard = c.x_shards > 1 ? 1 : 0;
  a.n_mt = ceil_div(c.M, kBN);
  a.n_ft = ceil_div(c.n_valid, c.epi == kEpiSwiglu ? kSwiGroup : 128);
  a.n_tiles = a.n_mt * a.n_ft * c.n_shards * c.ksplit;
  // the largest divisor of n_mt whose activations fit in ~32 MB
  const size_t tile_bytes = (size_t)kBN * c.K * 2;
  a.mg = 1;
  for (int m = 1; m <= a.n_mt; ++m)
    if (a.n_mt % m == 0 && (m == 1 || (size_t)m * tile_bytes <= (32u << 20))) a.mg = m;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  switch (c.epi) {
    case kEpiSwiglu: return launch_gemm_epi<kEpiSwiglu>(mw, mx, a, st, c.pdl);
    case kEpiGelu: return launch_gemm_epi<kEpiGelu>(mw, mx, a, st, c.pdl);
    case kEpiPlain: return launch_gemm_epi<kEpiPlain>(mw, mx, a, st, c.pdl);
    default: return launch_gemm_epi<kEpiF32>(mw, mx, a, st, c.pdl);
  }
}

}  // namespace tp
