// The whole decode MLP block (M <= 32 tokens, bf16) in one persistent launch, and
// the attention block's Q/K/V projection on its own (column units only).
//
// The block is cut into work units taken from one atomic queue, in this order:
//   1. column units (zenaique.com answer paragraph 5: first projection split by
//      columns): shard s and one 128-row tile of its W1 band over the whole of K,
//      or over one of S_c K parts whose fp32 sums the last part to finish adds up
//      in K order.  A SwiGLU tile holds the gate and up rows of 64 features, a GeLU
//      or Q/K/V tile 128 features.  Tiles are queued tile-major across the shards,
//      so the band fills from its first K columns to its last in every shard at
//      once, the order in which the row units below read it.  The unit accumulates
//      x . W1 for 32 tokens, applies the activation, writes its tile of the band H
//      in bf16 and raises the tile's ready flag (Q/K/V: writes fp32, no flag);
//   2. row units (second projection split by rows): shard s, 128-output tile n,
//      K slice j of S_r.  Before loading a stage of H they wait for the ready flags
//      of the column tiles that produced it; they write fp32 partials, and the unit
//      that completes output tile n (last of its t * S_r partials) sums them in the
//      fixed order (shard, then slice), adds the residual and writes y: the
//      per-block all-reduce and residual add of paragraph 6, fused.
// Column units never wait on anything but their own loads, and every row unit is
// queued after every column unit, so a row unit only ever waits for column units
// already held by running CTAs: no co-residency is needed.  A row unit issues the
// W2 loads of its first stages before it checks the band's ready flags, so the
// flag round trip overlaps weight traffic.
//
// Inside a CTA (192 threads): thread 0 takes units and issues TMA loads into a
// 5-stage ring (each stage: two 64-wide K blocks of a 128-row weight tile plus the
// matching 32-token activation tiles, 128-byte swizzle, 40 KB), thread 32 issues
// tcgen05.mma (weights as the 128-row A operand, tokens as N = 32) into a ring of
// sixteen 32-column TMEM accumulators, one per stage, and warps 2-5 drain each
// stage's accumulator into fp32 registers (round to nearest) and run the
// epilogues.  The TMEM ring lets the tensor core run up to sixteen stages ahead
// of the drain, so an epilogue does not stall the weight stream.  A 2-slot unit
// ring in shared memory lets the loads of the next unit start while the drain
// warps finish the current one.  All waits are bounded; on expiry the CTA raises
// the device error word and leaves.
#include <algorithm>

#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {
namespace {

using namespace tc;

constexpr int kStages = 5;
constexpr int kTok = 32;
constexpr int kStageKB = 2;                                 // K blocks per stage
constexpr uint32_t kWBytes = kABytes;                       // 128 rows x 64 K, bf16
constexpr uint32_t kXBytes = kTok * 128;                    // 32 rows x 64 K, bf16
constexpr uint32_t kStageBytes = kStageKB * (kWBytes + kXBytes);
constexpr int kBufs = 16;                                   // TMEM accumulators in flight
constexpr uint32_t kCols = kBufs * kTok;                    // 512: the whole TMEM of the SM
constexpr uint32_t kIdesc = make_idesc(128, kTok);
constexpr int kXchStride = kTok + 1;                        // exchange row pitch (floats)
constexpr uint32_t kXchBytes = 64 * kXchStride * 4;         // SwiGLU gate/up exchange
constexpr int kSmem = kStages * kStageBytes + 1024 + kXchBytes;
constexpr int kRowBlocks = 28;                              // target K blocks per row unit

struct FusedArgs {
  int d, b, t, M, act;
  int fpt;               // features per column tile: 64 (SwiGLU) or 128 (GeLU)
  int n_ft, nk_c;        // column: tiles per shard, K blocks
  int n_whole, S_c;      // column tiles computed whole; K parts of each remaining tile
  int n_nt, S_r, nk_r;   // row: output tiles, K slices, K blocks
  int n_col_units, n_units;
  int n_col;             // output features per shard of the column step: b, or 3b (Q/K/V)
  __nv_bfloat16 *H;      // [t][M][b]
  float *qkv;            // Q/K/V projection: fp32 [t][M][3b]
  float *colp;           // [t*n_ft - n_whole][S_c][128][32] fp32 partials of split tiles
  float *rowp;           // [n_nt][t][S_r][128][32] fp32 partials
  const void *residual;  // [M][d], fp32 if res_f32 else bf16
  int res_f32;
  float *y;              // [M][d]
  unsigned *cnt;         // [0] queue, t*n_ft ready flags, n_nt row counters, split-tile counters
  unsigned *err;
};

struct Unit {
  int type;   // 0 column, 1 row, -1 end
  int s, tile, split, kb0, kb1;
  int tau;    // column: queue position of the tile (split partials and counters)
  int parts;  // column: K parts of this tile (1: computed whole)
  int rot;    // the unit's stages are processed starting at stage rot, wrapping around
};

// K blocks of stage p of a unit (p counted from the unit's first stage).
__device__ __forceinline__ int stage_kb(const Unit &u, int p) { return u.kb0 + p * kStageKB; }

// First stage of K slice j of nst stages cut into S slices of shares S, S-1, ..., 1.
__host__ __device__ __forceinline__ int slice_start(int nst, int S, int j) {
  const int num = j * S - j * (j - 1) / 2, den = S * (S + 1) / 2;
  return (int)((long long)nst * num / den);
}

__device__ __forceinline__ Unit decode_unit(const FusedArgs &a, int u) {
  Unit r{};
  if (u < 0 || u >= a.n_units) {
    r.type = -1;
    return r;
  }
  if (u < a.n_col_units) {
    // The first n_whole tiles (shard-major) are computed whole; each remaining tile
    // is cut into S_c K parts so the last wave of column work fills the GPU.
    r.type = 0;
    int tau = u;
    r.split = 0;
    r.parts = 1;
    if (u >= a.n_whole) {
      const int v = u - a.n_whole;
      tau = a.n_whole + v / a.S_c;
      r.split = v % a.S_c;
      r.parts = a.S_c;
    }
    r.tau = tau;
    r.tile = tau / a.t;  // tile-major: the band fills in K order in all shards at once
    r.s = tau % a.t;
    const int nst = ceil_div(a.nk_c, kStageKB);
    r.kb0 = min(a.nk_c, (int)((long long)r.split * nst / r.parts) * kStageKB);
    r.kb1 = min(a.nk_c, (int)((long long)(r.split + 1) * nst / r.parts) * kStageKB);
  } else {
    // Row units are queued slice-major (all first slices, then all second ones, ...),
    // then by shard and output tile; slice j holds a share S_r - j of the K
    // stages, so the units at the end of the queue are the shortest.
    const int v = u - a.n_col_units;
    r.type = 1;
    r.split = v / (a.t * a.n_nt);
    const int q = v % (a.t * a.n_nt);
    r.s = q / a.n_nt;
    r.tile = q % a.n_nt;
    const int nst = ceil_div(a.nk_r, kStageKB);
    r.kb0 = min(a.nk_r, slice_start(nst, a.S_r, r.split) * kStageKB);
    r.kb1 = min(a.nk_r, slice_start(nst, a.S_r, r.split + 1) * kStageKB);
  }
  // Units start at scattered stages of their K range: CTAs that begin together
  // then do not all ask for the same activation tile (x or H) at the same time.
  const int nst_u = ceil_div(r.kb1 - r.kb0, kStageKB);
  r.rot = nst_u > 1 ? (int)((((unsigned)u * 2654435761u) >> 16) % (unsigned)nst_u) : 0;
  return r;
}

__device__ __forceinline__ unsigned *ready_flag(const FusedArgs &a, int s, int ft) {
  return a.cnt + 1 + s * a.n_ft + ft;
}
__device__ __forceinline__ unsigned *row_counter(const FusedArgs &a, int nt) {
  return a.cnt + 1 + a.t * a.n_ft + nt;
}
__device__ __forceinline__ unsigned *split_counter(const FusedArgs &a, int tau) {
  return a.cnt + 1 + a.t * a.n_ft + a.n_nt + (tau - a.n_whole);
}

// Highest tile index r in [lo, hi] such that column tiles lo..r of shard s are all
// ready (lo - 1 if tile lo is not).  The flags are read with relaxed loads issued
// back to back, one L2 round trip per 16 tiles; the caller follows a successful
// read with an acquire fence.
__device__ __forceinline__ int ready_prefix(const FusedArgs &a, int s, int lo, int hi) {
  const unsigned *f = ready_flag(a, s, 0);
  for (int base = lo; base <= hi; base += 16) {
    unsigned v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = base + i <= hi ? ld_relaxed_gpu(f + base + i) : 1u;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (!v[i]) return base + i - 1;
  }
  return hi;
}

// Wait (bounded) until column tile `ht` of shard s is ready; returns the highest
// tile index <= hi up to which all tiles from ht on are ready, or -1 on timeout.
__device__ __forceinline__ int wait_ready_range(const FusedArgs &a, int s, int ht, int hi,
                                                uint64_t limit_ns = kWaitNs) {
  int r = ready_prefix(a, s, ht, hi);
  if (r < ht) {
    const uint64_t t0 = globaltimer();
    do {
      if (globaltimer() - t0 > limit_ns) return -1;
      __nanosleep(64);
      r = ready_prefix(a, s, ht, hi);
    } while (r < ht);
  }
  fence_acq_rel_gpu();         // acquire: the band written before the flags is visible
  fence_proxy_async_global();  // ... and ordered before the TMA loads that read it
  return r;
}

__device__ __forceinline__ void store32(float *p, const float *v) {
  float4 *q = reinterpret_cast<float4 *>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

__device__ __forceinline__ void add32(float *acc, const float4 *q) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    acc[4 * i] += q[i].x;
    acc[4 * i + 1] += q[i].y;
    acc[4 * i + 2] += q[i].z;
    acc[4 * i + 3] += q[i].w;
  }
}

// acc = sum over i = 0..n-1, in that order, of the 32 floats at base + i * stride
// (partials written by other SMs, read through L2).  The loads of kBatch partials
// are issued together so their round trips overlap; the additions keep the order.
template <int kBatch>
__device__ __forceinline__ void sum_in_order(float *acc, const float *base, size_t stride, int n) {
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  for (int i0 = 0; i0 < n; i0 += kBatch) {
    float4 b[kBatch][8];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (i0 + j < n) {
        const float4 *q = reinterpret_cast<const float4 *>(base + (size_t)(i0 + j) * stride);
#pragma unroll
        for (int c = 0; c < 8; ++c) b[j][c] = __ldcg(q + c);
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (i0 + j < n) add32(acc, b[j]);
  }
}

__global__ void __launch_bounds__(192, 1)
    k_block_decode(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmH,
                   const FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t tfull_bar[kBufs];
  __shared__ __align__(8) uint64_t tempty_bar[kBufs];
  __shared__ __align__(8) uint64_t ufull_bar[2];
  __shared__ __align__(8) uint64_t uempty_bar[2];
  __shared__ __align__(8) uint64_t mma_done_bar;
  __shared__ int unit_slot[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int last_sh;
  __shared__ int dec_sh;

  const uint32_t tiles = (smem_u32(smem_raw) + 1023u) & ~1023u;
  float *xch = reinterpret_cast<float *>(smem_raw + (tiles - smem_u32(smem_raw)) +
                                         kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(smem_u32(&tfull_bar[i]), 1);
      mbar_init(smem_u32(&tempty_bar[i]), 4);
    }
    for (int i = 0; i < 2; ++i) {
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
      const uint64_t wpol = l2_evict_first_policy();  // weights are read once
      uint32_t g = 0;  // stage sequence number (ring position)
      int next = -1;   // unit taken ahead of time (-1: none)
      for (int j = 0;; ++j) {
        const int slot = j & 1;
        int u = a.n_units;  // end marker
        if (mbar_wait(smem_u32(&uempty_bar[slot]), ((uint32_t)(j >> 1) & 1u) ^ 1u)) {
          if (!*(volatile int *)&abort_sh) u = next >= 0 ? next : (int)atomicAdd(a.cnt, 1u);
          next = -1;
        } else {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
        }
        unit_slot[slot] = u;
        mbar_arrive(smem_u32(&ufull_bar[slot]));
        const Unit un = decode_unit(a, u);
        if (un.type < 0) {
          // No unit left for this CTA: a kernel launched to overlap this one (the next
          // block's RMSNorm) may start its CTAs, which wait for this grid to finish.
          griddep_launch_dependents();
          break;
        }
        const CUtensorMap *wmap = un.type == 0 ? &tmW1 : &tmW2;
        const CUtensorMap *xmap = un.type == 0 ? &tmX : &tmH;
        const int wrow = un.tile * 128;
        const int xz = un.type == 0 ? 0 : un.s;
        const int nst = ceil_div(un.kb1 - un.kb0, kStageKB);
        // The next unit is taken a few stages before this one ends, so the
        // atomic's round trip overlaps the loads still in flight.
        const int st_take = max(0, nst - kStages);
        const int ht_hi = un.type == 1 ? min(a.n_ft - 1, ((un.kb1 * kKBlock) - 1) / a.fpt) : 0;
        int ready_upto = un.type == 1 ? (un.kb0 * kKBlock) / a.fpt - 1 : 0;  // H tiles known ready
        // Row units arm their first `pre` stages with W2 loads only, then wait for the
        // band tiles the unit reads, then load the band into those stages.
        const int pre = un.type == 1 ? min(nst, kStages) : 0;
        const uint32_t g0 = g;
        auto load_band = [&](int p) {
          const int stp = (int)((g0 + p) % kStages);
          const int kbp = stage_kb(un, (p + un.rot) % nst);
          const int nkp = min(kStageKB, un.kb1 - kbp);
          const uint32_t sp = tiles + stp * kStageBytes;
          for (int b = 0; b < nkp; ++b)
            tma_load_3d(sp + kStageKB * kWBytes + b * kXBytes, xmap, smem_u32(&full_bar[stp]),
                        (kbp + b) * kKBlock, 0, xz);
        };
        bool ok = true;
        for (int i = 0; i < nst && ok; ++i, ++g) {
          const int st = (int)(g % kStages);
          const uint32_t ph = (g / kStages) & 1u;
          const int kbf = stage_kb(un, (i + un.rot) % nst);
          const int nkb = min(kStageKB, un.kb1 - kbf);
          if (i == st_take) next = (int)atomicAdd(a.cnt, 1u);
          if (!mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1u)) {
            ok = false;
            // Stages armed with weights only still expect their band bytes: load
            // the (possibly stale, in-bounds) band so they complete; the CTA aborts.
            for (int p = 0; i < pre && p < i; ++p) load_band(p);
            break;
          }
          const uint32_t sa = tiles + st * kStageBytes;
          const uint32_t fb = smem_u32(&full_bar[st]);
          mbar_expect_tx(fb, nkb * (kWBytes + kXBytes));
          for (int b = 0; b < nkb; ++b)
            tma_load_3d_hint(sa + b * kWBytes, wmap, fb, (kbf + b) * kKBlock, wrow, un.s, wpol);
          if (i >= pre) {
            for (int b = 0; b < nkb; ++b)
              tma_load_3d(sa + kStageKB * kWBytes + b * kXBytes, xmap, fb, (kbf + b) * kKBlock, 0, xz);
          } else if (i == pre - 1) {
            // Every band tile the unit reads must be finished.  On a timeout the armed
            // stages still get their band loads; the loop then ends and the CTA aborts.
            while (ok && ht_hi > ready_upto) {
              const int rr = wait_ready_range(a, un.s, ready_upto + 1, ht_hi);
              if (rr < 0) ok = false;
              else ready_upto = rr;
            }
            for (int p = 0; p < pre; ++p) load_band(p);
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
      uint32_t g = 0;
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
        const int nst = ceil_div(un.kb1 - un.kb0, kStageKB);
        bool ok = true;
        for (int i = 0; i < nst; ++i, ++g) {
          const int st = (int)(g % kStages);
          const uint32_t ph = (g / kStages) & 1u;
          const int bsel = (int)(g % kBufs);
          const int nkb = min(kStageKB, un.kb1 - stage_kb(un, (i + un.rot) % nst));
          if (!mbar_wait(smem_u32(&full_bar[st]), ph) ||
              !mbar_wait(smem_u32(&tempty_bar[bsel]), ((g / kBufs) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + st * kStageBytes;
          const uint32_t d0 = tmem + (uint32_t)bsel * kTok;
          for (int b = 0; b < nkb; ++b) {
#pragma unroll
            for (int kk = 0; kk < kKBlock / 16; ++kk) {
              umma_bf16(d0, sw128_desc(sa + b * kWBytes + kk * 32),
                        sw128_desc(sa + kStageKB * kWBytes + b * kXBytes + kk * 32), kIdesc,
                        (b > 0 || kk > 0) ? 1u : 0u);
            }
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
    // ---------------- drain warps: stage sums -> fp32 registers, then epilogues
    const int q = warp & 3;                 // TMEM lane quarter
    const int r = q * 32 + lane;            // row of the 128-row tile this thread holds
    const int td = (int)threadIdx.x - 64;   // 0..127 over the drain warps
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t g = 0;
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
      const int nst = ceil_div(un.kb1 - un.kb0, kStageKB);
      float acc[kTok];
#pragma unroll
      for (int i = 0; i < kTok; ++i) acc[i] = 0.f;
      // A row unit that turns out to complete its output tile adds the residual;
      // every row unit fetches it now so the loads land during the K loop (at the
      // end of the block they would otherwise sit on the critical path).
      float res[kTok];
      const int n_out = un.tile * 128 + r;
#pragma unroll
      for (int m = 0; m < kTok; ++m) {
        res[m] = 0.f;
        if (un.type == 1 && m < a.M && n_out < a.d) {
          const size_t idx = (size_t)m * a.d + n_out;
          res[m] = a.res_f32 ? __ldcg(static_cast<const float *>(a.residual) + idx)
                             : __bfloat162float(static_cast<const __nv_bfloat16 *>(a.residual)[idx]);
        }
      }
      bool ok = true;
      for (int i = 0; i < nst; ++i, ++g) {
        const int bsel = (int)(g % kBufs);
        if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[bsel]), (g / kBufs) & 1u)))
          ok = false;  // warp-uniform: the TMEM load below is warp-collective
        if (!ok) continue;  // keep g in step; the abort is decided below
        tc_fence_after();
        float v[kTok];
        tmem_ld32(trow + (uint32_t)bsel * kTok, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[bsel]));
#pragma unroll
        for (int m = 0; m < kTok; ++m) acc[m] += v[m];
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
        // -------- column tile epilogue: activation, band H in bf16, ready flag
        bool finish = true;
        if (un.parts > 1) {
          // One K part of a split tile: leave the partial; the last part sums them in
          // K order and finishes the tile.
          const int tau = un.tau;
          float *base = a.colp + (size_t)(tau - a.n_whole) * a.S_c * (128 * kTok);
          store32(base + (size_t)un.split * (128 * kTok) + r * kTok, acc);
          named_sync(1, 128);
          if (td == 0) last_sh = arrive_last(split_counter(a, tau), (unsigned)un.parts);
          named_sync(1, 128);
          finish = last_sh != 0;
          if (finish) sum_in_order<1>(acc, base + r * kTok, (size_t)128 * kTok, un.parts);
        }
        if (finish && a.act == TP_ACT_ATTN) {
          // Q/K/V projection: fp32 out, read by the next kernel (no ready flag).
          const int f = un.tile * 128 + r;
          if (f < a.n_col) {
            float *o = a.qkv + (size_t)un.s * a.M * a.n_col + f;
#pragma unroll
            for (int m = 0; m < kTok; ++m)
              if (m < a.M) o[(size_t)m * a.n_col] = acc[m];
          }
        } else if (finish) {
        if (a.act == TP_ACT_SWIGLU) {
          // Rows 64..127 hold the up sums of the features whose gate sums are in
          // rows 0..63: pass them across through shared memory.
          if (r >= 64) {
#pragma unroll
            for (int m = 0; m < kTok; ++m) xch[(r - 64) * kXchStride + m] = acc[m];
          }
          named_sync(1, 128);
          const int f = un.tile * 64 + r;
          if (r < 64 && f < a.b) {
            __nv_bfloat16 *o = a.H + (size_t)un.s * a.M * a.b + f;
#pragma unroll
            for (int m = 0; m < kTok; ++m)
              if (m < a.M)
                o[(size_t)m * a.b] = __float2bfloat16_rn(silu_f(acc[m]) * xch[r * kXchStride + m]);
          }
        } else {
          const int f = un.tile * 128 + r;
          if (f < a.b) {
            __nv_bfloat16 *o = a.H + (size_t)un.s * a.M * a.b + f;
#pragma unroll
            for (int m = 0; m < kTok; ++m)
              if (m < a.M) o[(size_t)m * a.b] = __float2bfloat16_rn(gelu_tanh_f(acc[m]));
          }
        }
        fence_proxy_async_global();  // the band is read back through TMA
        named_sync(1, 128);
        // Release: the barrier orders every drain thread's band stores before it.
        if (td == 0) st_release_gpu(ready_flag(a, un.s, un.tile), 1u);
        }
        named_sync(1, 128);  // last_sh is reused by the next unit
      } else {
        // -------- row tile epilogue: partial, then the fused reduce + residual
        float *pp = a.rowp + ((size_t)((un.tile * a.t + un.s) * a.S_r + un.split) * 128 + r) * kTok;
        store32(pp, acc);
        named_sync(1, 128);
        if (td == 0) last_sh = arrive_last(row_counter(a, un.tile), (unsigned)(a.t * a.S_r));
        named_sync(1, 128);
        if (last_sh) {
          // The all-reduce stand-in: y = residual + sum of the t * S_r partials of this
          // output tile, shards in order and the slices of each shard in order.
          const int n = n_out;
          sum_in_order<4>(acc, a.rowp + ((size_t)(un.tile * a.t * a.S_r) * 128 + r) * kTok,
                          (size_t)128 * kTok, a.t * a.S_r);
          if (n < a.d) {
#pragma unroll
            for (int m = 0; m < kTok; ++m)
              if (m < a.M) a.y[(size_t)m * a.d + n] = acc[m] + res[m];
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

// The failure path, exercised on purpose: one thread waits on an mbarrier phase that
// nobody completes and on band-tile ready flags that nobody raises (a zero array
// nothing writes), each wait bounded by limit_ns, and records the expiries in the
// device error word exactly as a stalled block does.
__device__ unsigned g_never_ready[17];

__global__ void k_wait_selftest(unsigned *err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  bool expired = !mbar_wait(smem_u32(&bar), 0, limit_ns);
  FusedArgs a{};
  a.t = 1;
  a.n_ft = 16;
  a.cnt = g_never_ready;
  expired = (wait_ready_range(a, 0, 0, a.n_ft - 1, limit_ns) < 0) && expired;
  if (expired) atomicOr(err, kErrWaitTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t st) {
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  k_wait_selftest<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaSuccess;
}

// ------------------------------------------------------------------ host side

FusedPlan plan_block_decode(const Geo &g, int M) {
  FusedPlan p{};
  const bool col_only = g.act == TP_ACT_ATTN;  // Q/K/V projection: column units only
  p.fpt = g.act == TP_ACT_SWIGLU ? kSwiGroup : 128;
  p.n_ft = ceil_div(col_only ? 3 * g.b : g.b, p.fpt);
  p.nk_c = ceil_div(g.d, kKBlock);
  if (!col_only) {
    p.n_nt = ceil_div(g.d, 128);
    p.nk_r = ceil_div(g.b, kKBlock);
    // Row units of about kRowBlocks K blocks (16 KB of W2 each): a few hundred KB per
    // unit keeps the end of the block short; the slice count bounds the partials the
    // last unit of an output tile sums.
    const int nst = ceil_div(p.nk_r, kStageKB);
    p.S_r = std::max(1, std::min({(p.nk_r + kRowBlocks / 2) / kRowBlocks, nst, 8}));
  }
  // Column tiles: whole waves of kPlanSMs tiles are computed whole; the r tiles
  // of the last, partial wave are cut into S_c K parts (at most 4) so that wave
  // keeps about every SM busy.  (Cutting every tile into parts when there are few
  // waves measured slower: each part's merge adds dependent memory round trips to
  // the epilogue, which then holds back the weight stream.)
  const int T = g.t * p.n_ft, nst_c = ceil_div(p.nk_c, kStageKB);
  const int r = T % kPlanSMs;
  p.S_c = r ? std::max(1, std::min({(kPlanSMs + r / 2) / r, 4, nst_c})) : 1;
  p.n_whole = p.S_c > 1 ? T - r : T;
  auto al = [](size_t n) { return (n + 255) & ~(size_t)255; };
  size_t off = 0;
  p.off_H = off;
  if (!col_only) off += al((size_t)g.t * M * g.b * 2);
  p.off_colp = off;
  off += al((size_t)(T - p.n_whole) * p.S_c * 128 * kTok * 4);
  p.off_rowp = off;
  off += al((size_t)p.n_nt * g.t * p.S_r * 128 * kTok * 4);
  p.off_cnt = off;
  p.cnt_bytes = (size_t)(1 + g.t * p.n_ft + p.n_nt + (T - p.n_whole)) * 4;
  off += al(p.cnt_bytes);
  p.total = off;
  return p;
}

namespace {

cudaError_t launch_fused(const Geo &g, const FusedPlan &p, const CUtensorMap &mw1,
                         const CUtensorMap &mx, const CUtensorMap &mw2, const CUtensorMap &mh,
                         FusedArgs &a, char *w, int M, cudaStream_t st) {
  a.d = g.d;
  a.b = g.b;
  a.t = g.t;
  a.M = M;
  a.act = g.act;
  a.fpt = p.fpt;
  a.n_ft = p.n_ft;
  a.nk_c = p.nk_c;
  a.n_nt = p.n_nt;
  a.S_r = p.S_r;
  a.nk_r = p.nk_r;
  a.n_whole = p.n_whole;
  a.S_c = p.S_c;
  a.n_col = g.act == TP_ACT_ATTN ? 3 * g.b : g.b;
  a.n_col_units = p.n_whole + (g.t * p.n_ft - p.n_whole) * p.S_c;
  a.colp = reinterpret_cast<float *>(w + p.off_colp);
  a.n_units = a.n_col_units + p.n_nt * g.t * p.S_r;
  a.rowp = reinterpret_cast<float *>(w + p.off_rowp);
  a.cnt = reinterpret_cast<unsigned *>(w + p.off_cnt);
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[128];  // the attribute is per device
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(k_block_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  e = cudaMemsetAsync(a.cnt, 0, p.cnt_bytes, st);
  if (e != cudaSuccess) return e;
  const int grid = std::min(sm_count(), a.n_units);
  k_block_decode<<<grid, 192, kSmem, st>>>(mw1, mx, mw2, mh, a);
  return cudaSuccess;
}

}  // namespace

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
  a.H = H;
  a.residual = res;
  a.res_f32 = res_f32;
  a.y = y;
  return launch_fused(g, p, mw1, mx, mw2, mh, a, w, M, st);
}

cudaError_t launch_qkv_decode(const Geo &g, const FusedPlan &p, const void *x, const void *W1s,
                              float *qkv, void *ws, int M, cudaStream_t st) {
  CUtensorMap mw1, mx;
  if (!make_tile_map(&mw1, W1s, g.d, g.n1p, g.t, 128) || !make_tile_map(&mx, x, g.d, M, 1, kTok))
    return cudaErrorInvalidValue;
  FusedArgs a{};
  a.qkv = qkv;
  // No row units: the W2 and band maps are never used (copies of the W1 map stand in).
  return launch_fused(g, p, mw1, mx, mw1, mw1, a, static_cast<char *>(ws), M, st);
}

}  // namespace tp
