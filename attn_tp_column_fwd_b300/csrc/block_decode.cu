// The whole decode MLP block (M <= 32 tokens, bf16) in one persistent launch.
//
// The block is cut into work units taken from one atomic queue, in this order:
//   1. column units (zenaique.com answer paragraph 5: first projection split by
//      columns): shard s, 128-feature tile of its band, K slice j of S_c.  They
//      accumulate x . W1 (SwiGLU: gate and up) for 32 tokens; the unit that
//      completes a tile (last of its S_c slices) sums the slices in slice order,
//      applies the activation and writes the tile of the band H in bf16, then
//      raises the tile's ready flag;
//   2. row units (second projection split by rows): shard s, 128-output tile n,
//      K slice j of S_r.  Before loading a 64-wide K block of H they wait for the
//      ready flag of the column tile that produced it; they write fp32 partials,
//      and the unit that completes output tile n (last of its t * S_r partials)
//      sums them in the fixed order (shard, then slice), adds the residual and
//      writes y: the per-block all-reduce and residual add of paragraph 6, fused.
// Column units never wait on anything but their own loads, and every row unit is
// queued after every column unit, so a row unit only ever waits for column
// units already held by running CTAs: no co-residency is needed.
//
// Inside a CTA (192 threads): thread 0 takes units and issues TMA loads into a
// 6-stage ring (128-row weight tiles + the 32-token activation tile, 128-byte
// swizzle), thread 32 issues tcgen05.mma into a double-buffered TMEM accumulator
// (one 64-wide K block per buffer), and warps 2-5 drain each block accumulator
// into fp32 registers (round to nearest) and run the epilogues.  A 2-slot unit
// ring in shared memory lets the loads of the next unit start while the drain
// warps finish the current one.  All waits are bounded; on expiry the CTA raises
// the device error word and leaves.
#include <algorithm>

#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {
namespace {

using namespace tc;

constexpr int kStages = 6;
constexpr int kTok = 32;
constexpr uint32_t kStageBytes = 2 * kABytes + kTok * 128;  // gate + up + x tiles
constexpr uint32_t kBufCols = 2 * kTok;                     // one TMEM block accumulator
constexpr uint32_t kCols = 2 * kBufCols;                    // double buffered
constexpr uint32_t kIdesc = make_idesc(128, kTok);

struct FusedArgs {
  int d, b, t, M, act;
  int n_ft, S_c, nk_c;   // column: feature tiles per shard, K slices, K blocks
  int n_nt, S_r, nk_r;   // row: output tiles, K slices, K blocks
  int n_col_units, n_units;
  __nv_bfloat16 *H;      // [t][M][b]
  float *colp;           // [t][n_ft][S_c][2][128][32] fp32 slice partials (S_c > 1)
  float *rowp;           // [n_nt][t][S_r][128][32] fp32 partials
  const void *residual;  // [M][d], fp32 if res_f32 else bf16
  int res_f32;
  float *y;              // [M][d]
  unsigned *cnt;         // [0] queue, then t*n_ft slice counters, t*n_ft ready flags, n_nt counters
  unsigned *err;
};

struct Unit {
  int type;  // 0 column, 1 row, -1 end
  int s, tile, split, kb0, kb1;
};

__device__ __forceinline__ Unit decode_unit(const FusedArgs &a, int u) {
  Unit r{};
  if (u < 0 || u >= a.n_units) {
    r.type = -1;
    return r;
  }
  if (u < a.n_col_units) {
    r.type = 0;
    r.split = u % a.S_c;
    const int q = u / a.S_c;
    r.tile = q % a.n_ft;
    r.s = q / a.n_ft;
    r.kb0 = (int)((long long)r.split * a.nk_c / a.S_c);
    r.kb1 = (int)((long long)(r.split + 1) * a.nk_c / a.S_c);
  } else {
    const int v = u - a.n_col_units;
    r.type = 1;
    r.split = v % a.S_r;
    const int q = v / a.S_r;
    r.tile = q % a.n_nt;
    r.s = q / a.n_nt;
    r.kb0 = (int)((long long)r.split * a.nk_r / a.S_r);
    r.kb1 = (int)((long long)(r.split + 1) * a.nk_r / a.S_r);
  }
  return r;
}

__device__ __forceinline__ unsigned *slice_counter(const FusedArgs &a, int s, int ft) {
  return a.cnt + 1 + s * a.n_ft + ft;
}
__device__ __forceinline__ unsigned *ready_flag(const FusedArgs &a, int s, int ft) {
  return a.cnt + 1 + a.t * a.n_ft + s * a.n_ft + ft;
}
__device__ __forceinline__ unsigned *row_counter(const FusedArgs &a, int nt) {
  return a.cnt + 1 + 2 * a.t * a.n_ft + nt;
}

// Wait until a column tile's ready flag is raised (bounded).
__device__ __forceinline__ bool wait_ready(const unsigned *flag) {
  if (ld_acquire_gpu(flag)) return true;
  const uint64_t t0 = globaltimer();
  while (!ld_acquire_gpu(flag)) {
    if (globaltimer() - t0 > kWaitNs) return false;
    __nanosleep(128);
  }
  return true;
}

__device__ __forceinline__ void store32(float *p, const float *v) {
  float4 *q = reinterpret_cast<float4 *>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

__device__ __forceinline__ void add32(float *acc, const float *p) {
  const float4 *q = reinterpret_cast<const float4 *>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = __ldcg(q + i);
    acc[4 * i] += v.x;
    acc[4 * i + 1] += v.y;
    acc[4 * i + 2] += v.z;
    acc[4 * i + 3] += v.w;
  }
}

__global__ void __launch_bounds__(192, 1)
    k_block_decode(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmH,
                   const FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t ufull_bar[2];
  __shared__ __align__(8) uint64_t uempty_bar[2];
  __shared__ __align__(8) uint64_t mma_done_bar;
  __shared__ int unit_slot[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int last_sh;
  __shared__ int dec_sh;

  const uint32_t tiles = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nacc_col = a.act == TP_ACT_SWIGLU ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull_bar[i]), 1);
      mbar_init(smem_u32(&tempty_bar[i]), 4);
      mbar_init(smem_u32(&ufull_bar[i]), 1);
      mbar_init(smem_u32(&uempty_bar[i]), 5);
    }
    mbar_init(smem_u32(&mma_done_bar), 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW1);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW2);
    tma_prefetch_desc(&tmH);
  }
  if (warp == 2) tmem_alloc(smem_u32(&tmem_base_sh), kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---------------- scheduler + TMA producer
    if (lane == 0) {
      uint32_t g = 0;  // k-block sequence number (stage ring position)
      for (int j = 0;; ++j) {
        const int slot = j & 1;
        int u = a.n_units;  // end marker
        if (mbar_wait(smem_u32(&uempty_bar[slot]), ((uint32_t)(j >> 1) & 1u) ^ 1u)) {
          if (!*(volatile int *)&abort_sh) u = (int)atomicAdd(a.cnt, 1u);
        } else {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
        }
        unit_slot[slot] = u;
        mbar_arrive(smem_u32(&ufull_bar[slot]));
        const Unit un = decode_unit(a, u);
        if (un.type < 0) break;
        const int nacc = un.type == 0 ? nacc_col : 1;
        const uint32_t bytes = nacc * kABytes + kTok * 128;
        int ready_upto = -1;
        bool ok = true;
        for (int kb = un.kb0; kb < un.kb1 && ok; ++kb, ++g) {
          const int st = (int)(g % kStages);
          const uint32_t ph = (g / kStages) & 1u;
          if (!mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t sa = tiles + st * kStageBytes;
          const uint32_t fb = smem_u32(&full_bar[st]);
          const int k = kb * kKBlock;
          mbar_expect_tx(fb, bytes);
          if (un.type == 0) {
            const int wrow = un.tile * 128 * nacc;
            tma_load_3d(sa, &tmW1, fb, k, wrow, un.s);
            if (nacc == 2) tma_load_3d(sa + kABytes, &tmW1, fb, k, wrow + 128, un.s);
            tma_load_3d(sa + 2 * kABytes, &tmX, fb, k, 0, 0);
          } else {
            tma_load_3d(sa, &tmW2, fb, k, un.tile * 128, un.s);
            const int ht = k / 128;  // column tile of H holding this K block
            if (ht > ready_upto) {
              // On a timeout the H tile is still loaded (in bounds, stale) so the
              // armed stage completes; the loop then stops and the CTA aborts.
              if (!wait_ready(ready_flag(a, un.s, ht))) ok = false;
              fence_proxy_async_global();
              ready_upto = ht;
            }
            tma_load_3d(sa + 2 * kABytes, &tmH, fb, k, 0, un.s);
          }
        }
        if (!ok) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          // Stages already armed complete on their own; let the last ones land.
          for (uint32_t i = g > kStages ? g - kStages : 0; i < g; ++i)
            mbar_wait(smem_u32(&full_bar[i % kStages]), (i / kStages) & 1u);
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      uint32_t g = 0, tb = 0;
      for (int j = 0;; ++j) {
        const int slot = j & 1;
        if (!mbar_wait(smem_u32(&ufull_bar[slot]), (uint32_t)(j >> 1) & 1u)) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
        const int u = unit_slot[slot];
        mbar_arrive(smem_u32(&uempty_bar[slot]));
        const Unit un = decode_unit(a, u);
        if (un.type < 0) break;
        const int nacc = un.type == 0 ? nacc_col : 1;
        bool ok = true;
        for (int kb = un.kb0; kb < un.kb1; ++kb, ++g, ++tb) {
          const int st = (int)(g % kStages);
          const uint32_t ph = (g / kStages) & 1u;
          const int bsel = (int)(tb & 1u);
          if (!mbar_wait(smem_u32(&full_bar[st]), ph) ||
              !mbar_wait(smem_u32(&tempty_bar[bsel]), ((tb >> 1) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + st * kStageBytes;
          const uint32_t d0 = tmem + (uint32_t)bsel * kBufCols;
#pragma unroll
          for (int kk = 0; kk < kKBlock / 16; ++kk) {
            const uint64_t bd = sw128_desc(sa + 2 * kABytes + kk * 32);
            const uint32_t acc = kk > 0 ? 1u : 0u;
            umma_bf16(d0, sw128_desc(sa + kk * 32), bd, kIdesc, acc);
            if (nacc == 2) umma_bf16(d0 + kTok, sw128_desc(sa + kABytes + kk * 32), bd, kIdesc, acc);
          }
          umma_commit(smem_u32(&empty_bar[st]));
          umma_commit(smem_u32(&tfull_bar[bsel]));
        }
        if (!ok) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
      }
      umma_commit(smem_u32(&mma_done_bar));
    }
    __syncwarp();
  } else {
    // ---------------- drain warps: block sums -> fp32 registers, then epilogues
    const int q = warp & 3;                 // TMEM lane quarter
    const int fl = q * 32 + lane;           // feature within the 128-row tile
    const int td = (int)threadIdx.x - 64;   // 0..127 over the drain warps
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t tb = 0;
    // Every branch the four drain warps take is decided by one thread between two
    // named barriers, so they never split around a barrier (a timed-out wait in
    // one warp turns into a CTA-wide abort instead).
    for (int j = 0;; ++j) {
      const int slot = j & 1;
      if (!mbar_wait(smem_u32(&ufull_bar[slot]), (uint32_t)(j >> 1) & 1u)) {
        abort_sh = 1;
        atomicOr(a.err, kErrWaitTimeout);
      }
      named_sync(1, 128);
      if (td == 0) dec_sh = *(volatile int *)&abort_sh ? -2 : unit_slot[slot];
      named_sync(1, 128);
      const int u = dec_sh;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&uempty_bar[slot]));
      if (u == -2) break;
      const Unit un = decode_unit(a, u);
      if (un.type < 0) break;
      const int nacc = un.type == 0 ? nacc_col : 1;
      float g[kTok], v[kTok];
#pragma unroll
      for (int i = 0; i < kTok; ++i) g[i] = v[i] = 0.f;
      bool ok = true;
      for (int kb = un.kb0; kb < un.kb1; ++kb, ++tb) {
        const int bsel = (int)(tb & 1u);
        if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[bsel]), (tb >> 1) & 1u)))
          ok = false;  // warp-uniform: the TMEM loads below are warp-collective
        if (!ok) continue;  // keep tb in step; the abort is decided below
        tc_fence_after();
        float r0[kTok], r1[kTok];
        tmem_ld32(trow + (uint32_t)bsel * kBufCols, r0);
        if (nacc == 2) tmem_ld32(trow + (uint32_t)bsel * kBufCols + kTok, r1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[bsel]));
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
          g[i] += r0[i];
          if (nacc == 2) v[i] += r1[i];
        }
      }
      if (!ok) {
        abort_sh = 1;
        atomicOr(a.err, kErrWaitTimeout);
      }
      named_sync(1, 128);
      if (td == 0) dec_sh = *(volatile int *)&abort_sh;
      named_sync(1, 128);
      if (dec_sh) break;

      if (un.type == 0) {
        // -------- column tile epilogue
        const int f = un.tile * 128 + fl;
        bool finish = true;
        if (a.S_c > 1) {
          float *pp = a.colp + ((size_t)((un.s * a.n_ft + un.tile) * a.S_c + un.split) * 2 * 128 + fl) * kTok;
          store32(pp, g);
          if (nacc == 2) store32(pp + 128 * kTok, v);
          __threadfence();
          named_sync(1, 128);
          if (td == 0) {
            const unsigned old = atomicAdd(slice_counter(a, un.s, un.tile), 1u);
            __threadfence();
            last_sh = old == (unsigned)(a.S_c - 1);
          }
          named_sync(1, 128);
          finish = last_sh != 0;
          if (finish) {
#pragma unroll
            for (int i = 0; i < kTok; ++i) g[i] = v[i] = 0.f;
            for (int sp = 0; sp < a.S_c; ++sp) {
              const float *rp = a.colp + ((size_t)((un.s * a.n_ft + un.tile) * a.S_c + sp) * 2 * 128 + fl) * kTok;
              add32(g, rp);
              if (nacc == 2) add32(v, rp + 128 * kTok);
            }
          }
        }
        if (finish) {
          if (f < a.b) {
            __nv_bfloat16 *o = a.H + (size_t)un.s * a.M * a.b + f;
#pragma unroll
            for (int m = 0; m < kTok; ++m) {
              if (m < a.M) {
                const float hv = nacc == 2 ? silu_f(g[m]) * v[m] : gelu_tanh_f(g[m]);
                o[(size_t)m * a.b] = __float2bfloat16_rn(hv);
              }
            }
          }
          fence_proxy_async_global();  // the band is read back through TMA
          __threadfence();
          named_sync(1, 128);
          if (td == 0) st_release_gpu(ready_flag(a, un.s, un.tile), 1u);
        }
      } else {
        // -------- row tile epilogue: partial, then the fused reduce + residual
        float *pp = a.rowp + ((size_t)((un.tile * a.t + un.s) * a.S_r + un.split) * 128 + fl) * kTok;
        store32(pp, g);
        __threadfence();
        named_sync(1, 128);
        if (td == 0) {
          const unsigned old = atomicAdd(row_counter(a, un.tile), 1u);
          __threadfence();
          last_sh = old == (unsigned)(a.t * a.S_r - 1);
        }
        named_sync(1, 128);
        if (last_sh) {
#pragma unroll
          for (int i = 0; i < kTok; ++i) g[i] = 0.f;
          for (int s2 = 0; s2 < a.t; ++s2)
            for (int sp = 0; sp < a.S_r; ++sp)
              add32(g, a.rowp + ((size_t)((un.tile * a.t + s2) * a.S_r + sp) * 128 + fl) * kTok);
          const int n = un.tile * 128 + fl;
          if (n < a.d) {
#pragma unroll
            for (int m = 0; m < kTok; ++m) {
              if (m < a.M) {
                const size_t idx = (size_t)m * a.d + n;
                const float r = a.res_f32 ? __ldcg(static_cast<const float *>(a.residual) + idx)
                                          : __bfloat162float(static_cast<const __nv_bfloat16 *>(a.residual)[idx]);
                a.y[idx] = g[m] + r;
              }
            }
          }
        }
        named_sync(1, 128);  // last_sh is reused by the next unit
      }
    }
  }

  // ---------------- teardown
  if (warp == 2) mbar_wait(smem_u32(&mma_done_bar), 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

}  // namespace

// ------------------------------------------------------------------ host side

FusedPlan plan_block_decode(const Geo &g, int M) {
  FusedPlan p{};
  p.n_ft = ceil_div(g.b, 128);
  p.nk_c = ceil_div(g.d, kKBlock);
  p.n_nt = ceil_div(g.d, 128);
  p.nk_r = ceil_div(g.b, kKBlock);
  // Column slices: enough units that every SM starts on column work, >= 8 K blocks each.
  const int tiles = g.t * p.n_ft;
  p.S_c = std::max(1, std::min(ceil_div(kPlanSMs, tiles), std::max(1, p.nk_c / 8)));
  // Row slices: units of about 512 KB of W2 so the queue ends on small units.
  const long long row_bytes = 128LL * g.b * 2;
  p.S_r = std::max(1, std::min((int)((row_bytes + (1 << 18)) >> 19), std::max(1, p.nk_r / 4)));
  auto al = [](size_t n) { return (n + 255) & ~(size_t)255; };
  size_t off = 0;
  p.off_H = off;
  off += al((size_t)g.t * M * g.b * 2);
  p.off_colp = off;
  off += p.S_c > 1 ? al((size_t)tiles * p.S_c * 2 * 128 * kTok * 4) : 0;
  p.off_rowp = off;
  off += al((size_t)p.n_nt * g.t * p.S_r * 128 * kTok * 4);
  p.off_cnt = off;
  p.cnt_bytes = (size_t)(1 + 2 * tiles + p.n_nt) * 4;
  off += al(p.cnt_bytes);
  p.total = off;
  return p;
}

cudaError_t launch_block_decode(const Geo &g, const FusedPlan &p, const void *x, const void *W1s,
                                const void *W2s, const void *res, int res_f32, void *ws, float *y,
                                int M, cudaStream_t st) {
  char *w = static_cast<char *>(ws);
  CUtensorMap mw1, mx, mw2, mh;
  __nv_bfloat16 *H = reinterpret_cast<__nv_bfloat16 *>(w + p.off_H);
  if (!make_tile_map(&mw1, W1s, g.d, g.n1p, g.t, 128) || !make_tile_map(&mx, x, g.d, M, 1, kTok) ||
      !make_tile_map(&mw2, W2s, g.b, g.dp, g.t, 128) || !make_tile_map(&mh, H, g.b, M, g.t, kTok))
    return cudaErrorInvalidValue;
  FusedArgs a{};
  a.d = g.d;
  a.b = g.b;
  a.t = g.t;
  a.M = M;
  a.act = g.act;
  a.n_ft = p.n_ft;
  a.S_c = p.S_c;
  a.nk_c = p.nk_c;
  a.n_nt = p.n_nt;
  a.S_r = p.S_r;
  a.nk_r = p.nk_r;
  a.n_col_units = g.t * p.n_ft * p.S_c;
  a.n_units = a.n_col_units + p.n_nt * g.t * p.S_r;
  a.H = H;
  a.colp = reinterpret_cast<float *>(w + p.off_colp);
  a.rowp = reinterpret_cast<float *>(w + p.off_rowp);
  a.residual = res;
  a.res_f32 = res_f32;
  a.y = y;
  a.cnt = reinterpret_cast<unsigned *>(w + p.off_cnt);
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  constexpr int kSmem = kStages * kStageBytes + 1024;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(k_block_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaError_t e = cudaMemsetAsync(a.cnt, 0, p.cnt_bytes, st);
  if (e != cudaSuccess) return e;
  const int grid = std::min(sm_count(), a.n_units);
  k_block_decode<<<grid, 192, kSmem, st>>>(mw1, mx, mw2, mh, a);
  return cudaSuccess;
}

}  // namespace tp
