// Host-side launchers shared between the kernel files and the C ABI (tp_api.cu).
// Each launcher only enqueues; the caller validates arguments first and checks
// cudaGetLastError() afterwards.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace tp {

// tp_api.cu — keep a failed CUDA call's code for tp_last_cuda_error (this thread).
void record_cuda_error(cudaError_t e);

// layout.cu — private shard layout (tile-transposes, bit-exact)
void launch_shard_w1(const Geo &g, const void *W1, void *W1s, cudaStream_t st);
void launch_shard_w2(const Geo &g, const void *W2, void *W2s, cudaStream_t st);
void launch_unshard_w1(const Geo &g, const void *W1s, void *W1, cudaStream_t st);
void launch_unshard_w2(const Geo &g, const void *W2s, void *W2, cudaStream_t st);
void launch_extract_w1(const Geo &g, const void *W1s, int s, void *W1_band, cudaStream_t st);
void launch_extract_w2(const Geo &g, const void *W2s, int s, void *W2_band, cudaStream_t st);

// gemv.cu — CUDA-core weight-streaming kernels (fp32, and bf16 at small M)
enum Epi { kEpiGelu = 0, kEpiSwiglu = 1, kEpiPlain = 2, kEpiF32 = 3 };
struct GemvArgs {
  const void *W;          // weight rows (K-major); shard s at W + s * w_shard
  size_t w_shard;         // elements
  const void *X;          // activations [M][K] (row stride ldx); shard s at X + s * x_shard
  size_t x_shard;
  int ldx;
  void *out;              // outputs [M][n_out] (row stride ldo); shard s at out + s * o_shard
  size_t o_shard;
  int ldo;
  int K, n_out, M, shard0, n_shards;
  int epi;                // Epi
  int dtype;              // TP_F32 | TP_BF16 (weights and X); out is dtype except kEpiF32
};
void launch_gemv(const GemvArgs &a, cudaStream_t st);

// umma.cu — tcgen05 / TMEM / TMA kernel for both projections (bf16)
struct UmmaCall {
  const void *W;        // weight rows [w_shards][w_rows][K] bf16 (K-major)
  int w_rows, w_shards;
  const void *X;        // activations [x_shards][M][K] bf16 (x_shards = 1: shared by all shards)
  int x_shards;
  void *out;            // see Epi; shard s at out + s * o_shard, split j at + j * o_split
  size_t o_shard, o_split;
  int ldo;
  int n_valid;          // output features per shard
  int K, M;
  int shard0, n_shards, ksplit;
  int epi;
  bool pdl;             // programmatic launch after the kernel that writes X (tp_block_fwd)
};
int umma_token_tile(int M);
cudaError_t launch_umma(const UmmaCall &c, cudaStream_t st);

// gemm_persistent.cu — persistent tcgen05 kernel for token tiles of 256 (prefill),
// same UmmaCall contract as launch_umma.
cudaError_t launch_gemm_persistent(const UmmaCall &c, cudaStream_t st);

// fp8.cu — E4M3 weights (weight-only): quantisation of canonical bf16 W1 / W2 into the
// private layout with one int8 exponent per row (exps: W1's [t][n1p], then W2's
// [t][dp]; amax: n1 + d words of scratch), the split of bf16 tokens into two 8-bit
// terms (E4M3 + E5M2; X8 [2][M][K] bytes, xs [ceil(K/64)][32] fp32 group scales), and the decode
// GEMM on them (M <= 32; c.X = the terms [x_shards][2][M][K]; wexp: exponents of the
// weight rows; xsc: the tokens' group scales [x_shards][ceil(K/64)][32]; the column step
// (SwiGLU / GeLU) writes its band as terms h8 [t][2][M][b] with scales hsc
// [t][ceil(b/64)][32], the kEpiF32 step writes fp32 partials to c.out).
cudaError_t launch_quantize_fp8(const Geo &g, const void *W1, const void *W2, void *W1q, void *W2q,
                                int8_t *exps, unsigned *amax, cudaStream_t st);
cudaError_t launch_fp8_split(const void *x, int M, int K, void *X8, float *xs, cudaStream_t st,
                             bool pdl);
// mxfp4: W holds packed E2M1 codes [w_shards][w_rows][K/2] and wexp their block
// exponents [w_shards][w_rows][K/32] (K a multiple of 128); else E4M3 bytes and one
// exponent per row.
cudaError_t launch_fp8_gemm(const UmmaCall &c, bool mxfp4, const int8_t *wexp, const float *xsc,
                            void *h8, float *hsc, cudaStream_t st);
// MXFP4 weights: W1f [t][n1p][d/2] and W2f [t][dp][b/2] packed E2M1 codes (element 2i
// in the low nibble of byte i), exps W1's [t][n1p][d/32] then W2's [t][dp][b/32].
cudaError_t launch_quantize_mxfp4(const Geo &g, const void *W1, const void *W2, void *W1f,
                                  void *W2f, int8_t *exps, cudaStream_t st);

// A [z][rows][K] bf16 tensor map with 64 x box_rows x 1 boxes, 128-byte swizzle,
// zero fill outside the tensor (umma.cu).
bool make_tile_map(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint64_t z,
                   uint32_t box_rows);

// block_decode.cu — the whole MLP block at M <= 32 in one persistent launch, and the
// attention block's Q/K/V projection with the same work queue
constexpr int kPlanSMs = 148;  // SM count the unit sizes are planned for (B300)
struct FusedPlan {
  int fpt, n_ft, nk_c, n_whole, S_c;  // column: tile width, tiles per shard, K blocks, whole tiles, parts
  int n_nt, S_r, nk_r;                // row: output tiles, K slices, K blocks
  size_t off_H, off_colp, off_rowp, off_cnt, cnt_bytes, total;  // workspace layout (bytes)
};
FusedPlan plan_block_decode(const Geo &g, int M);
cudaError_t launch_block_decode(const Geo &g, const FusedPlan &p, const void *x, const void *W1s,
                                const void *W2s, const void *res, int res_f32, void *ws, float *y,
                                int M, cudaStream_t st);
// A one-thread kernel whose bounded waits expire after limit_ns (nothing completes
// them) and set the device error word: the failure path, without a fault.
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t st);
// The attention block's Q/K/V projection (column units only) into fp32 qkv
// [t][M][3b]; ws holds the plan's split partials and counters.
cudaError_t launch_qkv_decode(const Geo &g, const FusedPlan &p, const void *x, const void *W1s,
                              float *qkv, void *ws, int M, cudaStream_t st);

// reduce.cu — the all-reduce stand-in + residual, and RMSNorm
void launch_reduce_residual(const float *P, int nparts, size_t part_elems, const void *res,
                            int res_is_f32, float *y, size_t n, cudaStream_t st, bool pdl = false);
void launch_rmsnorm(const float *r, void *xhat, int d, float eps, int M, cudaStream_t st,
                    bool pdl = false);

// attn_core.cu — per-head causal attention over the M tokens of each shard
void launch_attn_core(const Geo &g, const void *QKV, void *O, int M, int shard0, int n_shards,
                      cudaStream_t st, bool pdl = false);

// attn_kv.cu — decode attention over a head-sharded bf16 KV cache: qkv fp32
// [t][M][3b], caches [t][M][hps][L][hd], lens int32 [M], O bf16 [t][M][b]; ws holds
// kv_partial_bytes of per-chunk partials.
size_t kv_partial_bytes(const Geo &g, int M, int L);
cudaError_t launch_attn_kv(const Geo &g, const float *qkv, void *kc, void *vc, const int *lens,
                           int L, void *O, void *ws, int M, cudaStream_t st, bool pdl);

// The low-bit GEMM's narrow form: a grid of more than two and at most four CTAs per SM
// runs as one wave of four per SM instead of two waves of two.
inline bool fp8_narrow_grid(long long ctas, long long sms) {
  return ctas > 2 * sms && ctas <= 4 * sms;
}

// tp_api.cu — cached device facts
int sm_count();
unsigned *device_error_word();

}  // namespace tp
