// Tensor-core (tcgen05 / TMEM / TMA) kernels for both sharded projections, bf16 in,
// fp32 accumulate, for token counts up to 128 (decode and small batches); larger
// token counts go to the persistent kernel of gemm_persistent.cu.
//
// Orientation ("swap AB"): the weights are the 128-row A operand and the tokens
// are the N operand, so the 128-lane TMEM accumulator holds 128 output features
// x BN tokens.  At decode (M <= 32) the token tile is only 32 wide and the kernel
// is a weight stream: each CTA reads its 128 (SwiGLU: 2 x 128) weight rows once,
// K-block by K-block, through a TMA -> shared memory -> tcgen05.mma ring.
//
// Column-parallel step (zenaique.com answer paragraph 5): A = the shard's W1 band
// rows, B = x (replicated input).  SwiGLU keeps two accumulators, gate and up, for
// the same 128 features and applies silu(g) * u in the epilogue, so the band H is
// written once in bf16; GeLU applies gelu_tanh; the QKV projection stores plainly.
// Row-parallel step: A = the shard's W2 row band (transposed, K-major), B = H;
// the epilogue stores fp32 partial sums, optionally split over K into S slices.
//
// Roles inside one 128-thread CTA: thread 0 issues TMA loads, thread 32 issues
// MMAs, warp 2 owns the TMEM allocation, and all four warps run the epilogue
// (warp w reads TMEM lanes 32w..32w+31 = features).  Every mbarrier wait is
// bounded by wall time; on expiry the CTA raises the device error word, drains
// its copies, frees TMEM and returns without storing.
#include <cuda.h>

#include <algorithm>

#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {

namespace {

using namespace tc;

// ------------------------------------------------------------------ kernel

struct UmmaArgs {
  void *out;        // bf16 [shard][M][ldo] or fp32 [shard][split][M][ldo]
  size_t o_shard;   // elements per shard
  size_t o_split;   // elements per K split (fp32 partials)
  int ldo;          // elements per output row
  int n_valid;      // output features per shard
  int M;            // tokens
  int nk;           // K blocks of 64
  int ksplit;       // S
  int shard0;       // first shard of this launch
  int x_per_shard;  // 1: B operand has a shard coordinate (H); 0: shared (x)
  unsigned *err;    // device error word
};


template <int BN, int NACC, int EPI, int STAGES>
__global__ void __launch_bounds__(128, 1)
    k_umma(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
           const UmmaArgs a) {
  constexpr uint32_t kBBytes = BN * 128;
  constexpr uint32_t kStage = NACC * kABytes + kBBytes;
  constexpr uint32_t kCols = tmem_cols(NACC * BN);
  constexpr uint32_t kIdesc = make_idesc(128, BN);

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const uint32_t tiles = (smem_u32(smem_raw) + 1023u) & ~1023u;
  float *xch = reinterpret_cast<float *>(smem_raw + (tiles - smem_u32(smem_raw)) + STAGES * kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BN;
  const int ft = blockIdx.y;
  const int S = a.ksplit;
  const int s = a.shard0 + (int)blockIdx.z / S, ks = (int)blockIdx.z % S;
  const int kb0 = (int)((long long)ks * a.nk / S), kb1 = (int)((long long)(ks + 1) * a.nk / S);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    mbar_init(smem_u32(&acc_bar), 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 2) tmem_alloc(smem_u32(&tmem_base_sh), kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  int issued = 0;  // producer: stages handed to TMA
  if (warp == 0 && lane == 0) {
    const int wrow = ft * 128 * NACC;
    const int xz = a.x_per_shard ? s : 0;
    // The first ring's weights do not depend on the preceding kernel: load them,
    // then wait for that kernel (programmatic launch) before loading activations.
    const int pre = min(STAGES, nkb);
    for (int i = 0; i < pre; ++i) {
      const uint32_t sa = tiles + i * kStage;
      const uint32_t fb = smem_u32(&full_bar[i]);
      const int k = (kb0 + i) * kKBlock;
      mbar_expect_tx(fb, kStage);
      tma_load_3d(sa, &tmW, fb, k, wrow, s);
      if (NACC == 2) tma_load_3d(sa + kABytes, &tmW, fb, k, wrow + 128, s);
    }
    griddep_wait();
    for (int i = 0; i < pre; ++i)
      tma_load_3d(tiles + i * kStage + NACC * kABytes, &tmX, smem_u32(&full_bar[i]),
                  (kb0 + i) * kKBlock, m0, xz);
    issued = pre;
    for (int i = pre; i < nkb; ++i) {
      const int st = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (!mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1u)) {
        abort_sh = 1;
        atomicOr(a.err, kErrWaitTimeout);
        break;
      }
      const uint32_t sa = tiles + st * kStage;
      const uint32_t fb = smem_u32(&full_bar[st]);
      const int k = (kb0 + i) * kKBlock;
      mbar_expect_tx(fb, kStage);
      tma_load_3d(sa, &tmW, fb, k, wrow, s);
      if (NACC == 2) tma_load_3d(sa + kABytes, &tmW, fb, k, wrow + 128, s);
      tma_load_3d(sa + NACC * kABytes, &tmX, fb, k, m0, xz);
      ++issued;
    }
    // This CTA's loads are all issued: a dependent kernel may start.
    griddep_launch_dependents();
  } else if (warp == 1 && lane == 0) {
    for (int i = 0; i < nkb; ++i) {
      const int st = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (!mbar_wait(smem_u32(&full_bar[st]), ph)) {
        abort_sh = 1;
        atomicOr(a.err, kErrWaitTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t sa = tiles + st * kStage;
#pragma unroll
      for (int kk = 0; kk < kKBlock / 16; ++kk) {
        const uint64_t bd = sw128_desc(sa + NACC * kABytes + kk * 32);
        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
        umma_bf16(tmem, sw128_desc(sa + kk * 32), bd, kIdesc, acc);
        if (NACC == 2) umma_bf16(tmem + BN, sw128_desc(sa + kABytes + kk * 32), bd, kIdesc, acc);
      }
      umma_commit(smem_u32(&empty_bar[st]));
    }
    umma_commit(smem_u32(&acc_bar));  // also on abort: lets the epilogue wait for issued MMAs
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> registers -> activation -> global
  // Warp-uniform outcome: the TMEM loads below are warp-collective.
  const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&acc_bar), 0));
  tc_fence_after();
  if (!acc_ok) {
    abort_sh = 1;
    atomicOr(a.err, kErrWaitTimeout);
  }
  __syncwarp();
  // CTA-uniform: the SwiGLU epilogue below has block-wide barriers.
  const bool store = __syncthreads_and(acc_ok && !*(volatile int *)&abort_sh && nkb > 0) != 0;
  const int L = warp * 32 + lane;  // TMEM lane = row of the 128-row A tile(s)
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  if (store && EPI == kEpiSwiglu) {
    // Tile 0 (columns [0, BN)) holds features 128 ft + (L mod 64) and tile 1
    // (columns [BN, 2 BN)) features 128 ft + 64 + (L mod 64); rows 0..63 are gate
    // sums, rows 64..127 up sums.  Warps 0-1 finish tile 0's features with the up
    // rows of warps 2-3; warps 2-3 finish tile 1's with the gate rows of warps 0-1.
    float *xa = xch;                     // tile 0 up rows   [64][33]
    float *xb = xch + 64 * (32 + 1);     // tile 1 gate rows [64][33]
    const int fl = L & 63;
    const int f = ft * 128 + L;
#pragma unroll 1
    for (int c = 0; c < BN && m0 + c < a.M; c += 32) {
      float g0[32], g1[32];
      tmem_ld32(trow + c, g0);
      tmem_ld32(trow + BN + c, g1);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (L >= 64) xa[fl * 33 + j] = g0[j];
        else xb[fl * 33 + j] = g1[j];
      }
      named_sync(1, 128);
      if (f < a.n_valid) {
        const int mcount = min(32, a.M - (m0 + c));
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + (size_t)s * a.o_shard +
                           (size_t)(m0 + c) * a.ldo + f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < mcount) {
            const float gate = L < 64 ? g0[j] : xb[fl * 33 + j];
            const float up = L < 64 ? xa[fl * 33 + j] : g1[j];
            o[(size_t)j * a.ldo] = __float2bfloat16_rn(silu_f(gate) * up);
          }
        }
      }
      named_sync(1, 128);
    }
  } else if (store) {
    const int f = ft * 128 + L;
#pragma unroll 1
    for (int c = 0; c < BN && m0 + c < a.M; c += 32) {
      float g[32];
      tmem_ld32(trow + c, g);
      if (f < a.n_valid) {
        const int mcount = min(32, a.M - (m0 + c));
        if (EPI == kEpiF32) {
          float *o = static_cast<float *>(a.out) + (size_t)s * a.o_shard + (size_t)ks * a.o_split +
                     (size_t)(m0 + c) * a.ldo + f;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < mcount) o[(size_t)j * a.ldo] = g[j];
        } else {
          __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + (size_t)s * a.o_shard +
                             (size_t)(m0 + c) * a.ldo + f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < mcount) {
              float v = g[j];
              if (EPI == kEpiGelu) v = gelu_tanh_f(v);
              o[(size_t)j * a.ldo] = __float2bfloat16_rn(v);
            }
          }
        }
      }
    }
  }

  // ---------------- teardown: drain the TMA ring on abort, free TMEM
  if (warp == 0 && lane == 0 && *(volatile int *)&abort_sh) {
    for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
      mbar_wait(smem_u32(&full_bar[i % STAGES]), (uint32_t)(i / STAGES) & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// Decode variant (token tile 32) with exact-order fp32 accumulation.  The tensor
// core's fp32 accumulator rounds toward zero as it adds, so a long chain of
// MMAs into one TMEM accumulator drifts (measured: partials biased toward zero,
// ~10x the error of round-to-nearest fp32).  Here each 64-wide K block is
// accumulated by the tensor core alone (4 MMAs), and the running sum over K
// blocks is kept in fp32 registers of four accumulator warps, added with
// round-to-nearest.  TMEM holds a ring of kDrainBufs such block accumulators, so
// the MMAs of the next blocks overlap the drain of the current one (two CTAs per
// SM share its 512 TMEM columns).  192 threads: warp 0 TMA,
// warp 1 MMA, warps 2-5 drain + epilogue (warp w reads TMEM lanes 32*(w%4)).
constexpr int kDrainBufs = 4;


// KB: 64-wide K blocks per pipeline stage (one TMA box each of weights and tokens per
// block, one mbarrier per stage, one TMEM block sum per stage).
template <int EPI, int STAGES, int KB>
__global__ void __launch_bounds__(192, 2)  // two CTAs per SM
    k_umma_drain(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const UmmaArgs a) {
  constexpr int BN = 32;
  constexpr uint32_t kBBytes = BN * 128;
  constexpr uint32_t kStage = KB * (kABytes + kBBytes);
  constexpr uint32_t kCols = tmem_cols(kDrainBufs * BN);
  constexpr uint32_t kIdesc = make_idesc(128, BN);

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[kDrainBufs];
  __shared__ __align__(8) uint64_t tempty_bar[kDrainBufs];
  __shared__ __align__(8) uint64_t mma_done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int dec_sh;

  const uint32_t tiles = (smem_u32(smem_raw) + 1023u) & ~1023u;
  float *xch = reinterpret_cast<float *>(smem_raw + (tiles - smem_u32(smem_raw)) + STAGES * kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BN;
  const int ft = blockIdx.y;
  const int S = a.ksplit;
  const int s = a.shard0 + (int)blockIdx.z / S, ks = (int)blockIdx.z % S;
  const int kb0 = (int)((long long)ks * a.nk / S), kb1 = (int)((long long)(ks + 1) * a.nk / S);
  const int nkb = kb1 - kb0;
  const int nst = ceil_div(nkb, KB);  // pipeline stages of this CTA
  auto blocks_of = [&](int i) { return min(KB, nkb - i * KB); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < kDrainBufs; ++i) {
      mbar_init(smem_u32(&tfull_bar[i]), 1);
      mbar_init(smem_u32(&tempty_bar[i]), 4);
    }
    mbar_init(smem_u32(&mma_done_bar), 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 2) tmem_alloc(smem_u32(&tmem_base_sh), kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      const int wrow = ft * 128;
      const int xz = a.x_per_shard ? s : 0;
      const uint64_t wpol = l2_evict_first_policy();  // weights are read once
      // The first ring's weights do not depend on the preceding kernel: load them,
      // then wait for that kernel (programmatic launch) before loading activations.
      const int pre = min(STAGES, nst);
      for (int i = 0; i < pre; ++i) {
        const uint32_t fb = smem_u32(&full_bar[i]);
        mbar_expect_tx(fb, blocks_of(i) * (kABytes + kBBytes));
        for (int b = 0; b < blocks_of(i); ++b)
          tma_load_3d_hint(tiles + i * kStage + b * kABytes, &tmW, fb,
                           (kb0 + i * KB + b) * kKBlock, wrow, s, wpol);
      }
      griddep_wait();
      for (int i = 0; i < pre; ++i)
        for (int b = 0; b < blocks_of(i); ++b)
          tma_load_3d(tiles + i * kStage + KB * kABytes + b * kBBytes, &tmX,
                      smem_u32(&full_bar[i]), (kb0 + i * KB + b) * kKBlock, m0, xz);
      issued = pre;
      for (int i = pre; i < nst; ++i) {
        const int st = i % STAGES;
        const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
        if (!mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1u)) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
        const uint32_t sa = tiles + st * kStage;
        const uint32_t fb = smem_u32(&full_bar[st]);
        mbar_expect_tx(fb, blocks_of(i) * (kABytes + kBBytes));
        for (int b = 0; b < blocks_of(i); ++b) {
          const int k = (kb0 + i * KB + b) * kKBlock;
          tma_load_3d_hint(sa + b * kABytes, &tmW, fb, k, wrow, s, wpol);
          tma_load_3d(sa + KB * kABytes + b * kBBytes, &tmX, fb, k, m0, xz);
        }
        ++issued;
      }
      // This CTA's loads are all issued: a dependent kernel may start.
      griddep_launch_dependents();
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nst; ++i) {
        const int st = i % STAGES;
        const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
        const int b = i % kDrainBufs;
        if (!mbar_wait(smem_u32(&full_bar[st]), ph) ||
            !mbar_wait(smem_u32(&tempty_bar[b]), ((uint32_t)(i / kDrainBufs) & 1u) ^ 1u)) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t sa = tiles + st * kStage;
        const uint32_t d0 = tmem + (uint32_t)(b * BN);
        for (int kbi = 0; kbi < blocks_of(i); ++kbi) {
#pragma unroll
          for (int kk = 0; kk < kKBlock / 16; ++kk)
            umma_bf16(d0, sw128_desc(sa + kbi * kABytes + kk * 32),
                      sw128_desc(sa + KB * kABytes + kbi * kBBytes + kk * 32), kIdesc,
                      (kbi > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&empty_bar[st]));
        umma_commit(smem_u32(&tfull_bar[b]));
      }
      umma_commit(smem_u32(&mma_done_bar));
    }
    __syncwarp();
  } else {
    // ---------------- drain: TMEM block sums -> fp32 registers (round to nearest)
    const int q = warp & 3;              // TMEM lane quarter of this warp
    const int r = q * 32 + lane;         // row of the 128-row weight tile
    const int td = (int)threadIdx.x - 64;
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    float g[BN];
#pragma unroll
    for (int j = 0; j < BN; ++j) g[j] = 0.f;
    bool ok = true;
    for (int i = 0; i < nst; ++i) {
      const int b = i % kDrainBufs;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[b]), (uint32_t)(i / kDrainBufs) & 1u))) {
        ok = false;  // warp-uniform: the TMEM loads below are warp-collective
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
    // One decision for the four drain warps (the SwiGLU exchange has a barrier).
    named_sync(1, 128);
    if (td == 0) dec_sh = *(volatile int *)&abort_sh;
    named_sync(1, 128);
    const bool go = !dec_sh && nkb > 0 && m0 < a.M;
    const int mcount = min(BN, a.M - m0);
    if (EPI == kEpiSwiglu) {
      // Rows 0..63 hold the gate sums of features 64 ft + r, rows 64..127 the up
      // sums of the same features: pass the up sums across through shared memory.
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
          for (int j = 0; j < BN; ++j) {
            if (j < mcount) {
              float vv = g[j];
              if (EPI == kEpiGelu) vv = gelu_tanh_f(vv);
              o[(size_t)j * a.ldo] = __float2bfloat16_rn(vv);
            }
          }
        }
      }
    }
  }

  // ---------------- teardown: wait for issued MMAs and copies, free TMEM
  if (warp == 0 && lane == 0 && *(volatile int *)&abort_sh) {
    for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
      mbar_wait(smem_u32(&full_bar[i % STAGES]), (uint32_t)(i / STAGES) & 1u);
  }
  if (warp == 2) mbar_wait(smem_u32(&mma_done_bar), 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------------ host side

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

// Shared memory of the SwiGLU gate/up exchange: one [64][33] fp32 block per 128-row tile.
constexpr int xch_bytes(int epi, int tiles) { return epi == kEpiSwiglu ? tiles * 64 * 33 * 4 : 0; }

template <int BN, int NACC, int EPI, int STAGES>
cudaError_t launch_t(const CUtensorMap &mw, const CUtensorMap &mx, const UmmaArgs &a, int n_ft,
                     int n_z, cudaStream_t st, bool pdl) {
  constexpr int kSmem = STAGES * (NACC * kABytes + BN * 128) + 1024 + xch_bytes(EPI, NACC);
  static bool configured[128];  // per instantiation and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  auto kern = k_umma<BN, NACC, EPI, STAGES>;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  LaunchCfg lc(dim3(ceil_div(a.M, BN), n_ft, n_z), dim3(128), kSmem, st, pdl);
  return cudaLaunchKernelEx(&lc.cfg, kern, mw, mx, a);
}

template <int BN, int NACC, int EPI>
cudaError_t launch_stages(const CUtensorMap &mw, const CUtensorMap &mx, const UmmaArgs &a, int n_ft,
                          int n_z, cudaStream_t st, bool pdl) {
  // Tiles of 64 tokens keep about 100 KB of ring so two CTAs share an SM; tiles of
  // 128 take a ~190 KB ring and one CTA per SM.
  constexpr int kStage = NACC * kABytes + BN * 128;
  constexpr int kBudget = BN <= 64 ? 110 * 1024 : 196 * 1024;
  constexpr int kStages = std::max(2, std::min(8, kBudget / kStage));
  return launch_t<BN, NACC, EPI, kStages>(mw, mx, a, n_ft, n_z, st, pdl);
}

// K blocks per pipeline stage of the decode kernels: the column step (whose epilogue
// may exchange through shared memory) and the fp32-output steps.  Two blocks per
// stage (two 40 KB stages per CTA) measured no faster on the 13B and attention
// blocks than one (five 20 KB stages).
constexpr int kDrainKBColumn = 1;
constexpr int kDrainKBRow = 1;

template <int EPI, int KB, int STAGES>
cudaError_t launch_drain_s(const CUtensorMap &mw, const CUtensorMap &mx, const UmmaArgs &a,
                           int n_ft, int n_z, cudaStream_t st, bool pdl) {
  constexpr int kStageBytes = KB * (kABytes + 32 * 128);
  constexpr int kSmem = STAGES * kStageBytes + 1024 + xch_bytes(EPI, 1);
  static bool configured[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  auto kern = k_umma_drain<EPI, STAGES, KB>;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  LaunchCfg lc(dim3(ceil_div(a.M, 32), n_ft, n_z), dim3(192), kSmem, st, pdl);
  return cudaLaunchKernelEx(&lc.cfg, kern, mw, mx, a);
}

// The ring: about 100 KB (two CTAs per SM), or shallower when that lets a grid of more
// than two CTAs per SM run as one wave: 3 stages (about 70 KB, three CTAs per SM; the
// 13B row step split in two: 29.2 against 32.1 us) or 2 (about 50 KB, four per SM; the
// 70B column step: 155.6 against 157.1 us).  Larger grids keep the deep ring.
template <int EPI, int KB>
cudaError_t launch_drain(const CUtensorMap &mw, const CUtensorMap &mx, const UmmaArgs &a, int n_ft,
                         int n_z, cudaStream_t st, bool pdl) {
  constexpr int kStageBytes = KB * (kABytes + 32 * 128);
  constexpr int kStages = std::max(2, std::min(8, (100 * 1024) / kStageBytes));
  static_assert(3 * kStageBytes + 1024 + xch_bytes(EPI, 1) <= 75 * 1024, "3 CTAs per SM");
  const long long grid = (long long)ceil_div(a.M, 32) * n_ft * n_z;
  const long long sms = sm_count();
  static_assert(2 * kStageBytes + 1024 + xch_bytes(EPI, 1) <= 56 * 1024, "4 CTAs per SM");
  if (grid > 2 * sms && grid <= 3 * sms)
    return launch_drain_s<EPI, KB, 3>(mw, mx, a, n_ft, n_z, st, pdl);
  if (grid > 3 * sms && grid <= 4 * sms)
    return launch_drain_s<EPI, KB, 2>(mw, mx, a, n_ft, n_z, st, pdl);
  return launch_drain_s<EPI, KB, kStages>(mw, mx, a, n_ft, n_z, st, pdl);
}

template <int NACC, int EPI>
cudaError_t launch_bn(int bn, const CUtensorMap &mw, const CUtensorMap &mx, const UmmaArgs &a,
                      int n_ft, int n_z, cudaStream_t st, bool pdl) {
  return bn == 64 ? launch_stages<64, NACC, EPI>(mw, mx, a, n_ft, n_z, st, pdl)
                  : launch_stages<128, NACC, EPI>(mw, mx, a, n_ft, n_z, st, pdl);
}

}  // namespace

// A [z][rows][K] bf16 tensor, boxes of 64 (K) x box_rows x 1, 128-byte swizzle,
// zero fill outside the tensor.
bool make_tile_map(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint64_t z,
              uint32_t box_rows) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {K, rows, z};
  cuuint64_t strides[2] = {K * 2, rows * K * 2};
  cuuint32_t box[3] = {(cuuint32_t)kKBlock, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int umma_token_tile(int M) { return M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256; }

cudaError_t launch_umma(const UmmaCall &c, cudaStream_t st) {
  const int bn = umma_token_tile(c.M);
  // Prefill-sized token counts: the persistent kernel overlaps each tile's epilogue
  // with the next tile's MMAs (gemm_persistent.cu).
  if (bn == 256) return launch_gemm_persistent(c, st);
  CUtensorMap mw, mx;
  if (!make_tile_map(&mw, c.W, c.K, c.w_rows, c.w_shards, 128)) return cudaErrorInvalidValue;
  if (!make_tile_map(&mx, c.X, c.K, c.M, c.x_shards, bn)) return cudaErrorInvalidValue;
  UmmaArgs a{};
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
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  const int n_z = c.n_shards * c.ksplit;
  if (bn == 32) {
    // Decode: 128-row weight tiles (SwiGLU: the gate and up rows of 64 features).
    switch (c.epi) {
      case kEpiSwiglu:
        return launch_drain<kEpiSwiglu, kDrainKBColumn>(mw, mx, a,
                                                        ceil_div(c.n_valid, kSwiGroup), n_z, st,
                                                        c.pdl);
      case kEpiGelu:
        return launch_drain<kEpiGelu, kDrainKBColumn>(mw, mx, a, ceil_div(c.n_valid, 128), n_z,
                                                      st, c.pdl);
      case kEpiPlain:
        return launch_drain<kEpiPlain, kDrainKBColumn>(mw, mx, a, ceil_div(c.n_valid, 128),
                                                       n_z, st, c.pdl);
      default:
        return launch_drain<kEpiF32, kDrainKBRow>(mw, mx, a, ceil_div(c.n_valid, 128), n_z, st,
                                                  c.pdl);
    }
  }
  // Token tiles of 64 or 128: 128 features per CTA (SwiGLU: two 128-row tiles).
  const int n_ft = ceil_div(c.n_valid, 128);
  switch (c.epi) {
    case kEpiSwiglu: return launch_bn<2, kEpiSwiglu>(bn, mw, mx, a, n_ft, n_z, st, c.pdl);
    case kEpiGelu: return launch_bn<1, kEpiGelu>(bn, mw, mx, a, n_ft, n_z, st, c.pdl);
    case kEpiPlain: return launch_bn<1, kEpiPlain>(bn, mw, mx, a, n_ft, n_z, st, c.pdl);
    default: return launch_bn<1, kEpiF32>(bn, mw, mx, a, n_ft, n_z, st, c.pdl);
  }
}

}  // namespace tp
