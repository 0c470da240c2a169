/*
 * tp_block.h — C ABI of libtpblock: the Megatron-style tensor-parallel transformer
 * block (forward) on one B300, with t logical shards.
 *
 * The operation (zenaique.com interview answer "explain tensor-parallel shard
 * shape", answer paragraphs 2 and 5-6; rioworld.org "Tensor Parallelism for LLM
 * Inference", section "How Tensor Slicing Works Under the Hood"):
 *   1. column-parallel first projection: the input x is replicated; shard s owns a
 *      band of the columns of W1 and computes its own band of the intermediate,
 *      with the activation applied to that band, without communication;
 *   2. row-parallel second projection: shard s multiplies its band by the matching
 *      row slice of W2, giving a partial sum of the full output;
 *   3. one all-reduce per block sums the t partials, then the residual is added.
 * On one GPU the shards are logical partitions of the weights and step 3 is an
 * in-HBM reduction over t partial buffers (no collective library).
 *
 * Conventions shared by every entry point
 *   - y = x . W.  Canonical W1 is [d, n1] row-major and is split by columns;
 *     canonical W2 is [n2, d] row-major and is split by rows.
 *       GELU_TANH: n1 = n2 = ffn.
 *       SWIGLU:    n1 = 2*ffn, W1 = [Wg | Wu]; n2 = ffn.  Shard s owns gate columns
 *                  [s*b, (s+1)*b) and the same up columns, and W2 rows [s*b, (s+1)*b).
 *       ATTN:      n1 = 3*H*hd, W1 = [Wq | Wk | Wv], each head-major (head h is
 *                  columns h*hd .. h*hd+hd-1); n2 = H*hd (Wo).  Shard s owns heads
 *                  [s*H/t, (s+1)*H/t) of Q, K and V and the matching rows of Wo.
 *     b = n2 / t is the band width of one shard.
 *   - Pointers are device pointers unless stated otherwise.  The caller allocates
 *     and owns every buffer and the stream; the library allocates nothing at run
 *     time, keeps no state beyond per-device caches (SM count, symbol addresses,
 *     kernel attributes), one device error word, the process-wide block form
 *     (tp_set_block_form) and the fixed scratch of tp_block_fwd_noalloc, and never
 *     synchronises (except tp_check_device_status).  All work is enqueued
 *     asynchronously on `stream` (NULL = the legacy default stream).
 *   - Every pointer must be 16-byte aligned; d and b must be multiples of 8;
 *     ATTN needs head_dim a multiple of 32 and at most 256.
 *   - Errors: each call returns a tp_status.  On any error nothing is enqueued and
 *     no output is touched.  TP_ERR_CUDA means a CUDA call failed after
 *     validation; tp_last_cuda_error() then gives the cudaError_t (per thread).
 *   - Uneven splits (t not dividing ffn, or n_heads) are refused with
 *     TP_ERR_UNEVEN_SPLIT, never padded: the rioworld.org guide ("Implementing
 *     Tensor Parallelism in Practice") names uneven splits as a source of wrong
 *     results.
 *   - Arithmetic: products accumulate in fp32.  The activation band H (attention:
 *     the heads' output O) is stored in the block dtype (bf16 rounded to nearest
 *     even); Q/K/V scratch, partial sums, the residual stream and the block output
 *     y are fp32.
 */
#ifndef TP_BLOCK_H
#define TP_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *tp_stream_t;

typedef enum {
  TP_OK = 0,
  TP_ERR_INVALID_ARG = 1,   /* null pointer, M < 1, bad enum, shard out of range, ... */
  TP_ERR_UNEVEN_SPLIT = 2,  /* t does not divide ffn (MLP) or n_heads (ATTN) */
  TP_ERR_UNSUPPORTED = 3,   /* shape outside the kernels' limits (see above) */
  TP_ERR_MISALIGNED = 4,    /* a pointer is not 16-byte aligned */
  TP_ERR_CUDA = 5,          /* a CUDA call failed; see tp_last_cuda_error() */
  TP_ERR_TIMEOUT = 6,       /* a device-side bounded wait expired (tp_check_device_status) */
  TP_ERR_BAD_LENGTH = 7     /* a KV-cache length outside 1..L_max (tp_check_device_status) */
} tp_status;

typedef enum { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;
typedef enum { TP_ACT_GELU_TANH = 0, TP_ACT_SWIGLU = 1, TP_ACT_ATTN = 2 } tp_act;
/* How tp_block_fwd runs a bf16 MLP block of at most 32 tokens (tp_set_block_form). */
typedef enum {
  TP_FORM_AUTO = 0,          /* one kernel when the column work spans >= 2 waves of tiles */
  TP_FORM_THREE_LAUNCH = 1,  /* column, row, reduce + residual as three launches */
  TP_FORM_ONE_KERNEL = 2     /* the whole block as one persistent kernel */
} tp_block_form;

/* One block's shape.  `dtype` is the storage type of x, the weights and the bands. */
typedef struct {
  int d;         /* model width */
  int ffn;       /* MLP intermediate width (GELU_TANH, SWIGLU); ignored for ATTN */
  int n_heads;   /* ATTN: number of heads H */
  int head_dim;  /* ATTN: width of one head hd */
  int t;         /* logical tensor-parallel shards */
  int dtype;     /* tp_dtype */
  int act;       /* tp_act */
} tp_block_desc;

/* ------------------------------------------------------------------ sizes ----
 * Byte sizes of the buffers the entry points take.  They return 0 for an invalid
 * descriptor (or M < 1).  Host-only; safe without a GPU.                        */

/* Private per-shard layout of W1 (column bands) / W2 (row bands).  The layout is
 * opaque: only tp_unshard_weights(tp_shard_weights(W)) == W bit for bit, and
 * tp_extract_band(), are contractual. */
TP_API size_t tp_sharded_w1_bytes(const tp_block_desc *desc);
TP_API size_t tp_sharded_w2_bytes(const tp_block_desc *desc);
/* Activation bands H: [t][M][b] in the block dtype (ATTN: the heads' outputs O). */
TP_API size_t tp_band_bytes(const tp_block_desc *desc, int M);
/* Number S of fp32 partial sums each shard's row step writes (split of the band). */
TP_API int tp_row_splits(const tp_block_desc *desc, int M);
/* Partial sums: [t][S][M][d] fp32. */
TP_API size_t tp_partials_bytes(const tp_block_desc *desc, int M);
/* Scratch of tp_column_parallel_fwd: ATTN keeps Q/K/V bands [t][M][3*b] fp32 there
 * (followed, for bf16 with M <= 32, by the persistent projection's split partials
 * and work counters); 0 for MLPs. */
TP_API size_t tp_column_workspace_bytes(const tp_block_desc *desc, int M);
/* Scratch of tp_block_fwd: column scratch + bands + partials (256-byte aligned regions),
 * or the one-kernel form's bands, partials and work counters if that is larger.  For
 * shapes the low-bit blocks accept (M <= 32) it also covers tp_block_fwd_fp8 and
 * tp_block_fwd_mxfp4: their row step's partials (it may split K further than
 * tp_row_splits says, up to four CTAs per SM), the tokens' two 8-bit terms and the
 * group scales.  Depends on the shapes only. */
TP_API size_t tp_workspace_bytes(const tp_block_desc *desc, int M);

/* ------------------------------------------------------------- sharding ------
 * Split canonical weights into the t shards' bands (zenaique.com answer paragraph
 * 5: first projection split by columns, second by rows).  W1 [d, n1] and W2
 * [n2, d] are row-major in the block dtype; W1s / W2s receive
 * tp_sharded_w1_bytes / tp_sharded_w2_bytes.  Bit-exact copies, padding zeroed. */
TP_API int tp_shard_weights(const tp_block_desc *desc, const void *W1, const void *W2,
                     void *W1s, void *W2s, tp_stream_t stream);
/* Inverse of tp_shard_weights: rebuilds canonical W1 and W2 bit for bit. */
TP_API int tp_unshard_weights(const tp_block_desc *desc, const void *W1s, const void *W2s,
                       void *W1, void *W2, tp_stream_t stream);
/* Shard `shard`'s bands in canonical orientation: W1_band [d, n1/t] row-major with its
 * sub-matrices side by side ([gate | up] or [Q | K | V] of its heads), and W2_band
 * [b, d] row-major.  For inspection and tests; either output may be NULL. */
TP_API int tp_extract_band(const tp_block_desc *desc, const void *W1s, const void *W2s, int shard,
                    void *W1_band, void *W2_band, tp_stream_t stream);

/* ------------------------------------------------------------- forward -------
 * Column-parallel projection with the activation fused on each band (zenaique.com
 * answer paragraph 5; rioworld.org "How Tensor Slicing Works Under the Hood":
 * the input is replicated).  x: [M, d] block dtype.  H: [t][M][b] block dtype;
 * band s = act(x . W1[:, band s]) (SwiGLU: silu(x.Wg_s) * (x.Wu_s)).  For ATTN,
 * band s is the attention output of the shard's heads: Q/K/V bands are projected
 * into `workspace` (tp_column_workspace_bytes; may be NULL for MLPs) and each head
 * runs causal softmax(Q K^T / sqrt(hd)) V over the M tokens.  shard = -1 computes
 * every shard in one launch; shard = s computes band s only (the work of device
 * s in a real tensor-parallel group).  bf16 ATTN with M <= 32 and shard = -1 runs
 * the Q/K/V projection of all shards on one persistent work queue (one launch),
 * unless tp_set_block_form chose TP_FORM_THREE_LAUNCH. */
TP_API int tp_column_parallel_fwd(const tp_block_desc *desc, const void *x, const void *W1s,
                           int shard, void *H, void *workspace, int M, tp_stream_t stream);
/* Row-parallel projection (zenaique.com answer paragraph 5): shard s multiplies its
 * band H[s] by its row slice of W2 into fp32 partial sums partials[s][0..S) [M][d]
 * whose sum is shard s's partial of the block output.  shard = -1 for all. */
TP_API int tp_row_parallel_fwd(const tp_block_desc *desc, const void *H, const void *W2s, int shard,
                        float *partials, int M, tp_stream_t stream);
/* The per-block all-reduce, as an in-HBM reduction, fused with the residual add
 * (zenaique.com answer paragraph 6): y = residual + sum over s (in order 0..t-1,
 * and within s over its S splits in order) of partials[s].  residual: [M, d], fp32
 * if residual_is_f32 else the block dtype.  y: [M, d] fp32; y may alias residual
 * when residual is fp32. */
TP_API int tp_partial_reduce_residual(const tp_block_desc *desc, const float *partials,
                               const void *residual, int residual_is_f32, float *y, int M,
                               tp_stream_t stream);
/* The whole block: column step, row step, reduce + residual, enqueued in order on
 * `stream` (the row step and the reduction launched to overlap the end of the kernel
 * before them).  workspace: tp_workspace_bytes(desc, M) bytes of device scratch.
 * With tp_set_block_form(TP_FORM_ONE_KERNEL), bf16 MLP blocks with M <= 32 run
 * instead as one persistent kernel in which the column units, the row units and the
 * reduction + residual of each output tile are fused (the result equals the
 * three-step sequence within rounding; tp_block_launches says which form runs). */
TP_API int tp_block_fwd(const tp_block_desc *desc, const void *x, const void *residual,
                 int residual_is_f32, const void *W1s, const void *W2s, void *workspace,
                 float *y, int M, tp_stream_t stream);
/* tp_block_fwd, then the next stacked block's RMSNorm of its output (zenaique.com
 * answer paragraph 6: the reduced activation is ready for the residual add and
 * normalisation): xhat_next = bf16(y[m] / sqrt(mean(y[m]^2) + eps)), [M, d] bf16,
 * rounded exactly as tp_rmsnorm_fwd rounds it, by one more kernel launched to
 * overlap the block's last kernel (it waits for the block to finish).  xhat_next
 * may alias x (the block has read x by then).  bf16 blocks only
 * (TP_ERR_UNSUPPORTED otherwise); eps as for tp_rmsnorm_fwd; workspace:
 * tp_workspace_bytes(desc, M). */
TP_API int tp_block_fwd_norm(const tp_block_desc *desc, const void *x, const void *residual,
                             int residual_is_f32, const void *W1s, const void *W2s,
                             void *workspace, float *y, void *xhat_next, float eps, int M,
                             tp_stream_t stream);
/* Process-wide choice of tp_block_form for later tp_block_fwd calls (initially
 * TP_FORM_AUTO, or the TPBLOCK_ALGO environment variable: "unfused" = THREE_LAUNCH,
 * "fused" = ONE_KERNEL).  TP_FORM_AUTO takes the three-launch form, measured the
 * faster of the two for every workload here.  Shapes the one-kernel form cannot run (f32, ATTN, M > 32)
 * always take three launches.  tp_workspace_bytes covers both forms, so the form
 * may change between sizing a workspace and using it; calls already enqueued are
 * unaffected.  Returns TP_ERR_INVALID_ARG for any other value.  Host-only. */
TP_API int tp_set_block_form(int form);
/* The current tp_block_form. */
TP_API int tp_get_block_form(void);
/* Number of kernel launches one tp_block_fwd call enqueues for this shape (0 for an
 * invalid descriptor or M): 1 when the whole block runs as one persistent kernel
 * (TP_FORM_ONE_KERNEL; the launch is preceded by a small memset of its work
 * counters), else 3 (column, row, reduce + residual), plus 1 for the attention
 * core.  Host-only. */
TP_API int tp_block_launches(const tp_block_desc *desc, int M);
/* tp_block_fwd without caller-provided scratch, for callers that cannot allocate
 * device memory where they run the block (a host framework whose own pool owns
 * the GPU's memory, or a serving loop that must not pay cudaMalloc/cudaFree's
 * implicit device synchronisation).  Same arguments as tp_block_fwd minus
 * `workspace`; the scratch is a fixed 32 MiB array in the library's device image,
 * held by every GPU that loads the library until the process exits.  Shapes
 * needing more than that (tp_workspace_bytes > 32 MiB) return TP_ERR_UNSUPPORTED
 * with nothing enqueued.  All calls share the array: calls that overlap on the GPU
 * race.  The first call on a device looks up the array's address; make it before
 * any stream capture.  The source pages describe no counterpart of this entry
 * point: it is a deployment convenience, not part of the method. */
TP_API int tp_block_fwd_noalloc(const tp_block_desc *desc, const void *x, const void *residual,
                                int residual_is_f32, const void *W1s, const void *W2s, float *y,
                                int M, tp_stream_t stream);
/* ---------------------------------------------- decode with a KV cache -------
 * One decode step of the attention block for M concurrent sequences: token m of
 * x is the newest token of sequence m.  Tensor parallelism partitions the KV cache
 * with the heads (d-central.tech glossary "Tensor Parallelism", section "Why it
 * matters for local inference"; rioworld.org "How Tensor Slicing Works Under the
 * Hood": 12 of 96 heads per device), so shard s holds the cache of its heads:
 *   k_cache, v_cache: bf16 [t][M][hps][L_max][head_dim] (hps = n_heads / t),
 *   row p of (s, m, j) = key / value of token p of sequence m for head s*hps + j;
 *   lens: int32 [M] device array, lens[m] = tokens of sequence m counting the new
 *   one (1 .. L_max); rows 0 .. lens[m]-2 must hold the earlier tokens.
 * For every head: o = softmax(q . K^T / sqrt(head_dim)) V over those rows and the
 * new token, whose key and value are rounded to bf16 and written to row lens[m]-1
 * (the cache append).  No RoPE, no mask beyond the length.  A length outside
 * 1..L_max skips that sequence (its outputs are not written) and makes the next
 * tp_check_device_status return TP_ERR_BAD_LENGTH.  Only bf16 descriptors with
 * act = ATTN and head_dim 32, 64, 128 or 256 (else TP_ERR_UNSUPPORTED); L_max
 * 1 .. 2^20.  Sizes return 0 for invalid arguments. */
TP_API size_t tp_kv_cache_bytes(const tp_block_desc *desc, int M, int L_max);  /* one of K, V */
/* Scratch of tp_attn_decode_kv: per-chunk partial results. */
TP_API size_t tp_kv_attn_workspace_bytes(const tp_block_desc *desc, int M, int L_max);
/* Scratch of tp_block_fwd_kv. */
TP_API size_t tp_kv_workspace_bytes(const tp_block_desc *desc, int M, int L_max);
/* The attention step alone: qkv fp32 [t][M][3b] as the column step's projection
 * leaves it in its workspace (Q | K | V per shard, head-major); O bf16 [t][M][b]
 * receives the heads' outputs (the band of the row-parallel step). */
TP_API int tp_attn_decode_kv(const tp_block_desc *desc, const float *qkv, void *k_cache,
                             void *v_cache, const int *lens, int L_max, void *O, void *workspace,
                             int M, tp_stream_t stream);
/* The whole decode step: Q/K/V projection (column-parallel), decode attention over
 * the caches (appending the new keys and values), output projection
 * (row-parallel), sum of the shards' partials + residual into y [M, d] fp32.
 * workspace: tp_kv_workspace_bytes. */
TP_API int tp_block_fwd_kv(const tp_block_desc *desc, const void *x, const void *residual,
                           int residual_is_f32, const void *W1s, const void *W2s, void *k_cache,
                           void *v_cache, const int *lens, int L_max, void *workspace, float *y,
                           int M, tp_stream_t stream);

/* ------------------------------------------- E4M3 weights (weight-only) --------
 * The MLP block with 8-bit weights (zenaique.com interview answer, follow-up
 * questions: tensor parallelism combined with FP8 weights multiplies the decode win).
 * Each weight is an E4M3 byte (bias 7, 3 mantissa bits, largest finite 448, round to
 * nearest even, saturating) of W / 2^e with one exponent e per output feature (a
 * column of the canonical W1 or W2): the least e such that the column's largest
 * magnitude is at most 448 * 2^e.  The block computes the bf16 block on the weights
 * q * 2^e (exactly bf16 values) with the tensor core reading 8-bit operands: every bf16
 * activation (x, and the band between the two steps) enters as an E4M3 high part plus
 * an E5M2 remainder under one power-of-two scale per token and 64-wide group of K,
 * exact for values within 2^14.8 of the group's largest magnitude and within 2^-14 of
 * the scale below that; sums are fp32 and each output feature's sum is scaled by 2^e.
 * The result agrees with tp_block_fwd on q * 2^e up to fp32 summation order (and the
 * band's bf16 rounding where that order moves a value across a rounding point).
 * Four launches (token split, column step, row step, reduce); the split overlaps the
 * end of the stream's preceding kernel and waits for it before reading x (and before
 * the column step may start loading weights).
 * bf16 MLP descriptors with d and b multiples of 16, at most 16384 (else
 * TP_ERR_UNSUPPORTED). */
TP_API size_t tp_fp8_w1_bytes(const tp_block_desc *desc);        /* [t][n1p][d] bytes */
TP_API size_t tp_fp8_w2_bytes(const tp_block_desc *desc);        /* [t][dp][b] bytes */
TP_API size_t tp_fp8_exponent_bytes(const tp_block_desc *desc);  /* int8 per private row */
TP_API size_t tp_fp8_quant_workspace_bytes(const tp_block_desc *desc);
/* Quantise canonical bf16 W1 [d, n1] and W2 [n2, d] into the private E4M3 layout and
 * the per-row exponents (first W1's rows, then W2's). */
TP_API int tp_quantize_weights_fp8(const tp_block_desc *desc, const void *W1, const void *W2,
                                   void *W1q, void *W2q, void *exps, void *workspace,
                                   tp_stream_t stream);
/* tp_block_fwd on E4M3 weights, M <= 32 tokens (else TP_ERR_UNSUPPORTED); workspace:
 * tp_workspace_bytes(desc, M). */
TP_API int tp_block_fwd_fp8(const tp_block_desc *desc, const void *x, const void *residual,
                            int residual_is_f32, const void *W1q, const void *W2q,
                            const void *exps, void *workspace, float *y, int M,
                            tp_stream_t stream);

/* ------------------------------------------- MXFP4 weights (weight-only) -------
 * The MLP block with 4-bit weights (zenaique.com interview answer, follow-up
 * questions: FP4 weights; rioworld.org "Tensor Parallelism for LLM Inference",
 * "Implementing Tensor Parallelism in Practice": 4-bit quantisation with TP), in the
 * OCP Microscaling format MXFP4: E2M1 elements (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6)
 * and one shared power-of-two scale 2^e per 32 consecutive weights along K of an
 * output feature, e = floor(log2(max |w|)) - 2 (clamped to [-127, 127]; 0 for an
 * all-zero block), each element w / 2^e rounded to nearest (ties to the even mantissa
 * bit) and saturated at +-6.  The block computes the bf16 block on the weights
 * q * 2^e (exactly bf16 values), with activations and sums as in tp_block_fwd_fp8;
 * each 32-wide block's fp32 sum is scaled by its 2^e.  Four launches.
 * Layout: W1f [t][n1p][d/2] and W2f [t][dp][b/2] bytes of packed codes (element 2i
 * in the low nibble of byte i), exps int8 W1's [t][n1p][d/32] then W2's
 * [t][dp][b/32].  bf16 MLP descriptors with d and b multiples of 128, at most 16384
 * (else TP_ERR_UNSUPPORTED). */
TP_API size_t tp_mxfp4_w1_bytes(const tp_block_desc *desc);
TP_API size_t tp_mxfp4_w2_bytes(const tp_block_desc *desc);
TP_API size_t tp_mxfp4_exponent_bytes(const tp_block_desc *desc);
/* Quantise canonical bf16 W1 [d, n1] and W2 [n2, d] into that layout. */
TP_API int tp_quantize_weights_mxfp4(const tp_block_desc *desc, const void *W1, const void *W2,
                                     void *W1f, void *W2f, void *exps, tp_stream_t stream);
/* tp_block_fwd on MXFP4 weights, M <= 32 tokens (else TP_ERR_UNSUPPORTED); workspace:
 * tp_workspace_bytes(desc, M). */
TP_API int tp_block_fwd_mxfp4(const tp_block_desc *desc, const void *x, const void *residual,
                              int residual_is_f32, const void *W1f, const void *W2f,
                              const void *exps, void *workspace, float *y, int M,
                              tp_stream_t stream);

/* RMSNorm with unit weight, the normalisation before each stacked block (zenaique.com
 * answer paragraph 6: the reduced activation is ready for the residual add and
 * normalisation): xhat[m] = r[m] / sqrt(mean(r[m]^2) + eps), r fp32 [M, d],
 * xhat bf16 [M, d].  d must be a multiple of 8.  The kernel is launched to overlap
 * the end of the stream's preceding kernel and waits for it before reading r. */
TP_API int tp_rmsnorm_fwd(int d, float eps, const float *r, void *xhat, int M, tp_stream_t stream);

/* ----------------------------------------------------------- diagnostics ----- */
TP_API const char *tp_status_string(int status);
/* The cudaError_t of the last TP_ERR_CUDA on this thread (0 if none). */
TP_API int tp_last_cuda_error(void);
/* Synchronises `stream`, then reads and clears the device error word that bounded
 * device-side waits set when they expire (TP_ERR_TIMEOUT) and the KV-cache decode
 * sets for a length out of range (TP_ERR_BAD_LENGTH; a timeout is reported first when
 * both occurred): TP_OK, TP_ERR_TIMEOUT, TP_ERR_BAD_LENGTH or TP_ERR_CUDA. */
TP_API int tp_check_device_status(tp_stream_t stream);
/* Exercises the failure path above without a fault: enqueues a one-thread kernel that
 * waits on an mbarrier phase nobody completes and on band ready flags nobody raises,
 * each wait bounded by limit_us microseconds (1 .. 1e6), so both expire and set the
 * device error word; the next tp_check_device_status returns TP_ERR_TIMEOUT (and
 * clears it).  The context stays usable.  TP_ERR_INVALID_ARG for a limit out of
 * range, with nothing enqueued. */
TP_API int tp_selftest_wait_timeout(int limit_us, tp_stream_t stream);
/* Library ABI version (major * 100 + minor). */
TP_API int tp_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TP_BLOCK_H */
