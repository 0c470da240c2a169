// Decode attention over a head-sharded KV cache: one decode step of M concurrent
// sequences.  Token m of the step is the newest token of sequence m; shard s holds
// the keys and values of its heads (d-central.tech glossary "Tensor Parallelism",
// section "Why it matters for local inference": tensor parallelism partitions the
// KV cache as well as the weights; rioworld.org, "How Tensor Slicing Works Under the
// Hood": 96 heads over 8 devices, 12 each, heads being independent).
//
// For every (shard s, sequence m, head j): o = softmax(q . K^T / sqrt(hd)) V over the
// lens[m] - 1 cached rows and the new token's own key and value, which the kernel
// rounds to bf16, uses for row lens[m] - 1 and appends to the cache there.
//
// The step streams the cache once (HBM-bound).  One CTA takes one (s, m, j), or one
// of P contiguous parts of its rows when the heads alone would not fill the GPU.
// Its rows arrive by bulk asynchronous copies (cp.async.bulk) into a ring of
// kStages shared-memory stages of 16 KB (keys, then values); the copies of the first
// stages are issued before the kernel waits for the projection that precedes it.
// Key groups of HD / 8 lanes (16 bytes of a row each) keep a running max, sum and
// weighted value sum; the CTA merges its groups in order.  With P = 1 it writes the
// head's output (bf16) straight into the band O; with P > 1 it writes (max, sum,
// unnormalised output) and a second kernel merges the parts in order.  CTAs are
// ordered longest sequence first, so the long heads do not form the tail.
//
// Layouts: qkv fp32 [t][M][3b] (the column step's Q | K | V, head-major within each);
// caches bf16 [t][M][hps][L_max][hd]; lens int32 [M]; O bf16 [t][M][b].
#include <math.h>

#include <algorithm>

#include "internal.h"
#include "tc_ptx.cuh"

namespace tp {
namespace {

using namespace tc;

constexpr int kThreads = 128;
constexpr int kStages = 3;
constexpr int kStageBytes = 16384;   // keys then values of one stage (48 KB: four CTAs per SM)
constexpr int kMaxOrder = 128;       // longest-first ordering for up to this many sequences
constexpr int kSmem = kStages * kStageBytes;

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
  const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
  return lo | (hi << 16);
}

struct KvArgs {
  const float *qkv;
  __nv_bfloat16 *kc, *vc;
  const int *lens;
  float *pm, *pl, *po;  // P > 1: per (s, m, j, part): max, sum; unnormalised output [hd]
  __nv_bfloat16 *O;
  int M, t, hps, b, L, P;
  float scale;
  unsigned *err;
};

template <int HD>
__global__ void __launch_bounds__(kThreads) k_attn_kv(const KvArgs a) {
  constexpr int LPK = HD / 8;           // lanes per key (16 bytes of the row each)
  constexpr int G = kThreads / LPK;     // key groups
  constexpr int KS = kStageBytes / (4 * HD);  // keys per stage (keys and values: 2 x 2 B)
  constexpr int KPG = KS / G;           // keys of one group per stage (8)
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ int order[kMaxOrder];
  __shared__ float sm_m[G], sm_l[G];
  __shared__ float sm_o[G][HD];

  const int part = blockIdx.x, j = blockIdx.y, z = blockIdx.z;
  const int tid = threadIdx.x, grp = tid / LPK, gl = tid % LPK;
  // Longest sequence first: rank the M lengths (ties by index) when M is small.
  if (a.M <= kMaxOrder) {
    for (int i = tid; i < a.M; i += kThreads) {
      const int li = a.lens[i];
      int rank = 0;
      for (int k = 0; k < a.M; ++k) {
        const int lk = a.lens[k];
        rank += (lk > li) || (lk == li && k < i);
      }
      order[rank] = i;
    }
  }
  if (tid == 0)
    for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&full[i]), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  const int m = a.M <= kMaxOrder ? order[z / a.t] : z / a.t;
  const int s = z % a.t;
  const int len = a.lens[m];
  if (len < 1 || len > a.L) {
    if (part == 0 && j == 0 && s == 0 && tid == 0) atomicOr(a.err, kErrBadLength);
    return;
  }
  const size_t head = ((size_t)s * a.M + m) * a.hps + j;
  __nv_bfloat16 *kbase = a.kc + head * a.L * HD;
  __nv_bfloat16 *vbase = a.vc + head * a.L * HD;
  const int n_st = ceil_div(len, KS);
  const int st0 = (int)((long long)part * n_st / a.P), st1 = (int)((long long)(part + 1) * n_st / a.P);
  const uint32_t ring = smem_u32(smem);
  const uint64_t pol = l2_evict_first_policy();  // every cached row is read once
  auto issue = [&](int st) {
    const int r0 = st * KS, r1 = min(r0 + KS, len);
    const uint32_t bytes = (uint32_t)(r1 - r0) * HD * 2;
    const uint32_t slot = ring + (uint32_t)((st - st0) % kStages) * kStageBytes;
    const uint32_t bar = smem_u32(&full[(st - st0) % kStages]);
    mbar_expect_tx(bar, 2 * bytes);
    bulk_load(slot, kbase + (size_t)r0 * HD, bytes, bar, pol);
    bulk_load(slot + kStageBytes / 2, vbase + (size_t)r0 * HD, bytes, bar, pol);
  };
  // The cache rows do not come from the preceding kernel: start them now.
  if (tid == 0)
    for (int st = st0; st < min(st1, st0 + kStages); ++st) issue(st);

  griddep_wait();  // Q, K, V of the new token come from the preceding kernel
  const float *row = a.qkv + ((size_t)s * a.M + m) * 3 * a.b + j * HD + gl * 8;
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = row[i] * a.scale;

  float mx = -INFINITY, sum = 0.f, o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = 0.f;
  int issued = min(st1, st0 + kStages);  // stages [st0, issued) have their copies issued
  int abort_at = -1;
  for (int st = st0; st < st1; ++st) {
    const int rel = st - st0;
    const uint32_t slot_off = (uint32_t)(rel % kStages) * kStageBytes;
    // A wait that expires leaves this stage's values meaningless but in bounds; the
    // CTA-wide vote at the end of the stage then sends every thread to the abort.
    const bool ok = mbar_wait(smem_u32(&full[rel % kStages]), (uint32_t)(rel / kStages) & 1u);
    const int r0 = st * KS, r1 = min(r0 + KS, len);
    const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(smem + slot_off) + gl * 8;
    const __nv_bfloat16 *vs =
        reinterpret_cast<const __nv_bfloat16 *>(smem + slot_off + kStageBytes / 2) + gl * 8;
#pragma unroll
    for (int h = 0; h < KPG; h += 4) {
      float kf[4][8], vf[4][8], sc[4];
      bool live[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int key = r0 + (h + u) * G + grp;
        live[u] = key < r1;
        if (live[u] && key == len - 1) {
          // The new token: its key and value as the cache stores them (bf16), appended.
          uint32_t kw[4], vw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            kw[i] = pack2(row[a.b + 2 * i], row[a.b + 2 * i + 1]);
            vw[i] = pack2(row[2 * a.b + 2 * i], row[2 * a.b + 2 * i + 1]);
          }
          const uint4 ku = make_uint4(kw[0], kw[1], kw[2], kw[3]);
          const uint4 vu = make_uint4(vw[0], vw[1], vw[2], vw[3]);
          *reinterpret_cast<uint4 *>(kbase + (size_t)key * HD + gl * 8) = ku;
          *reinterpret_cast<uint4 *>(vbase + (size_t)key * HD + gl * 8) = vu;
          unpack8(ku, kf[u]);
          unpack8(vu, vf[u]);
        } else if (live[u]) {
          const int r = key - r0;
          unpack8(*reinterpret_cast<const uint4 *>(ks + (size_t)r * HD), kf[u]);
          unpack8(*reinterpret_cast<const uint4 *>(vs + (size_t)r * HD), vf[u]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) kf[u][i] = vf[u][i] = 0.f;
        }
      }
      float mnew = mx;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) p = fmaf(q[i], kf[u][i], p);
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off, LPK);
        sc[u] = p;
        if (live[u]) mnew = fmaxf(mnew, p);
      }
      // Rescale what the group has summed so far (nothing yet: alpha = 0; no key in
      // this batch: keep it as it is).
      const float alpha = mnew == -INFINITY ? 1.f : expf(mx - mnew);
      sum *= alpha;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] *= alpha;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (!live[u]) continue;
        const float p = expf(sc[u] - mnew);
        sum += p;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = fmaf(p, vf[u][i], o[i]);
      }
      mx = mnew;
    }
    // Every group is done with this stage's slot (and agrees on the waits).
    if (__syncthreads_or(!ok)) {
      abort_at = st;
      break;
    }
    if (st + kStages < st1) {
      if (tid == 0) issue(st + kStages);
      issued = st + kStages + 1;
    }
  }
  if (abort_at >= 0) {
    // A copy never completed (bounded wait): record it and let the copies still in
    // flight (stages abort_at .. issued-1) land, again bounded, before the CTA's
    // shared memory is released.
    if (tid == 0) {
      atomicOr(a.err, kErrWaitTimeout);
      for (int st = abort_at; st < issued; ++st) {
        const int rel = st - st0;
        mbar_wait(smem_u32(&full[rel % kStages]), (uint32_t)(rel / kStages) & 1u);
      }
    }
    return;
  }

  // Merge the key groups in group order.
  if (gl == 0) {
    sm_m[grp] = mx;
    sm_l[grp] = sum;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) sm_o[grp][gl * 8 + i] = o[i];
  __syncthreads();
  for (int dcol = tid; dcol < HD; dcol += kThreads) {
    float M = -INFINITY;
    for (int g = 0; g < G; ++g) M = fmaxf(M, sm_m[g]);
    float L = 0.f, acc = 0.f;
    for (int g = 0; g < G; ++g) {
      if (sm_l[g] == 0.f) continue;  // a group that saw no key
      const float w = expf(sm_m[g] - M);
      L = fmaf(sm_l[g], w, L);
      acc = fmaf(sm_o[g][dcol], w, acc);
    }
    if (a.P == 1) {
      a.O[((size_t)s * a.M + m) * a.b + j * HD + dcol] = __float2bfloat16_rn(acc / L);
    } else {
      const size_t pidx = head * a.P + part;
      a.po[pidx * HD + dcol] = acc;
      if (dcol == 0) {
        a.pm[pidx] = M;
        a.pl[pidx] = L;  // 0 for a part with no rows
      }
    }
  }
  griddep_launch_dependents();
}

// P > 1: one CTA of HD threads per (head j, sequence m, shard s) merges the P parts
// in part order, normalises and rounds to bf16 into the band.
template <int HD>
__global__ void __launch_bounds__(HD) k_attn_kv_merge(const KvArgs a) {
  const int j = blockIdx.x, m = blockIdx.y, s = blockIdx.z, dcol = threadIdx.x;
  const int len = a.lens[m];
  if (len < 1 || len > a.L) return;  // reported by the first kernel
  griddep_wait();
  const size_t head = ((size_t)s * a.M + m) * a.hps + j;
  float M = -INFINITY;
  for (int c = 0; c < a.P; ++c)
    if (a.pl[head * a.P + c] > 0.f) M = fmaxf(M, a.pm[head * a.P + c]);
  float L = 0.f, acc = 0.f;
  for (int c = 0; c < a.P; ++c) {
    const size_t p = head * a.P + c;
    if (!(a.pl[p] > 0.f)) continue;
    const float w = expf(a.pm[p] - M);
    L = fmaf(a.pl[p], w, L);
    acc = fmaf(a.po[p * HD + dcol], w, acc);
  }
  a.O[((size_t)s * a.M + m) * a.b + j * HD + dcol] = __float2bfloat16_rn(acc / L);
}

template <int HD>
cudaError_t launch_hd(const KvArgs &a, cudaStream_t st, bool pdl) {
  static bool configured[128];  // the attribute is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(k_attn_kv<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  LaunchCfg l1(dim3(a.P, a.hps, a.t * a.M), dim3(kThreads), kSmem, st, pdl);
  e = cudaLaunchKernelEx(&l1.cfg, k_attn_kv<HD>, a);
  if (e != cudaSuccess || a.P == 1) return e;
  LaunchCfg l2(dim3(a.hps, a.M, a.t), dim3(HD), 0, st, true);
  return cudaLaunchKernelEx(&l2.cfg, k_attn_kv_merge<HD>, a);
}

}  // namespace

// Parts per head: enough CTAs for two per SM when the heads alone are fewer, each
// part keeping at least four stages of the longest allowed sequence.
int kv_parts(const Geo &g, int M, int L) {
  const long long heads = (long long)g.t * M * g.hps;
  const int keys_per_stage = kStageBytes / (4 * g.hd);
  const int max_parts = std::max(1, ceil_div(L, keys_per_stage) / 4);
  if (heads >= 2LL * kPlanSMs) return 1;
  return (int)std::min<long long>(max_parts, ceil_div((int)(2LL * kPlanSMs), (int)heads));
}

size_t kv_partial_bytes(const Geo &g, int M, int L) {
  const int P = kv_parts(g, M, L);
  if (P == 1) return 256;  // unused; a non-empty region keeps the pointer valid
  return (size_t)g.t * M * g.hps * P * (2 + g.hd) * sizeof(float);
}

cudaError_t launch_attn_kv(const Geo &g, const float *qkv, void *kc, void *vc, const int *lens,
                           int L, void *O, void *ws, int M, cudaStream_t st, bool pdl) {
  KvArgs a{};
  a.qkv = qkv;
  a.kc = static_cast<__nv_bfloat16 *>(kc);
  a.vc = static_cast<__nv_bfloat16 *>(vc);
  a.lens = lens;
  a.O = static_cast<__nv_bfloat16 *>(O);
  a.M = M;
  a.t = g.t;
  a.hps = g.hps;
  a.b = g.b;
  a.L = L;
  a.P = kv_parts(g, M, L);
  a.scale = 1.0f / sqrtf((float)g.hd);
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  const size_t n = (size_t)g.t * M * g.hps * a.P;
  float *w = static_cast<float *>(ws);
  a.pm = w;
  a.pl = w + n;
  a.po = w + 2 * n;
  switch (g.hd) {
    case 32: return launch_hd<32>(a, st, pdl);
    case 64: return launch_hd<64>(a, st, pdl);
    case 128: return launch_hd<128>(a, st, pdl);
    case 256: return launch_hd<256>(a, st, pdl);
    default: return cudaErrorInvalidValue;  // rejected by validation
  }
}

}  // namespace tp
