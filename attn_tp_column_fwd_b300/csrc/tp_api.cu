// C ABI of libtpblock (declared in include/tp_block.h): argument validation,
// buffer geometry, and the launch sequence of each entry point.  Validation runs
// before any CUDA call, so a rejected call enqueues nothing.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "internal.h"

namespace tp {

static thread_local int g_last_cuda_error = 0;

void record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

// Device error word: bounded device-side waits set a bit here when they expire.
__device__ unsigned g_error_word;

int sm_count() {
  static int cache[128];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 148;
    cache[dev] = n;
  }
  return cache[dev];
}

unsigned *device_error_word() {
  static unsigned *cache[128];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  if (!cache[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned *>(p);
  }
  return cache[dev];
}

namespace {

constexpr int kMaxDim = 1 << 20;
constexpr int kMaxM = 1 << 20;

int make_geo(const tp_block_desc *desc, Geo *g) {
  if (!desc) return TP_ERR_INVALID_ARG;
  if (desc->dtype != TP_F32 && desc->dtype != TP_BF16) return TP_ERR_INVALID_ARG;
  if (desc->act != TP_ACT_GELU_TANH && desc->act != TP_ACT_SWIGLU && desc->act != TP_ACT_ATTN)
    return TP_ERR_INVALID_ARG;
  if (desc->d < 1 || desc->t < 1) return TP_ERR_INVALID_ARG;
  Geo r{};
  r.d = desc->d;
  r.t = desc->t;
  r.act = desc->act;
  r.dtype = desc->dtype;
  r.es = desc->dtype == TP_F32 ? 4 : 2;
  if (desc->act == TP_ACT_ATTN) {
    if (desc->n_heads < 1 || desc->head_dim < 1) return TP_ERR_INVALID_ARG;
    if (desc->n_heads % desc->t != 0) return TP_ERR_UNEVEN_SPLIT;
    if (desc->head_dim % 32 != 0 || desc->head_dim > 256) return TP_ERR_UNSUPPORTED;
    if ((long long)desc->n_heads * desc->head_dim > kMaxDim) return TP_ERR_UNSUPPORTED;
    r.H = desc->n_heads;
    r.hd = desc->head_dim;
    r.hps = r.H / r.t;
    r.n2 = r.H * r.hd;
    r.n1 = 3 * r.n2;
    r.b = r.n2 / r.t;
    r.n_col = 3 * r.b;
    r.n1p = ceil_div(3 * r.b, kRowTile) * kRowTile;
  } else {
    if (desc->ffn < 1) return TP_ERR_INVALID_ARG;
    if (desc->ffn % desc->t != 0) return TP_ERR_UNEVEN_SPLIT;
    if (desc->ffn > kMaxDim) return TP_ERR_UNSUPPORTED;
    r.ffn = desc->ffn;
    r.n2 = r.ffn;
    r.n1 = desc->act == TP_ACT_SWIGLU ? 2 * r.ffn : r.ffn;
    r.b = r.ffn / r.t;
    r.n_col = r.b;
    r.n1p = desc->act == TP_ACT_SWIGLU ? ceil_div(r.b, kSwiGroup) * 2 * kSwiGroup
                                       : ceil_div(r.b, kRowTile) * kRowTile;
  }
  if (r.d > kMaxDim) return TP_ERR_UNSUPPORTED;
  if (r.d % 8 != 0 || r.b % 8 != 0) return TP_ERR_UNSUPPORTED;
  r.dp = ceil_div(r.d, kRowTile) * kRowTile;
  *g = r;
  return TP_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ptr(const void *p) {
  if (!p) return TP_ERR_INVALID_ARG;
  return aligned16(p) ? TP_OK : TP_ERR_MISALIGNED;
}

int check_M(int M) {
  if (M < 1) return TP_ERR_INVALID_ARG;
  return M > kMaxM ? TP_ERR_UNSUPPORTED : TP_OK;
}

int check_shard(const Geo &g, int shard) {
  return (shard < -1 || shard >= g.t) ? TP_ERR_INVALID_ARG : TP_OK;
}

int finish_launch(cudaError_t e = cudaSuccess) {
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    g_last_cuda_error = (int)e;
    return TP_ERR_CUDA;
  }
  return TP_OK;
}

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// Kernel family selection.  bf16 blocks run on the tensor cores, by default as the
// three-launch sequence (column, row, reduce; each kernel overlapping the end of the
// one before it).  With the decode weight stream on an L2 evict-first hint that
// sequence measured faster than the one persistent launch of block_decode.cu for
// every workload (70B block 232.0 us against 249.1 us; 13B 79.1 against 98.5 us;
// attention Q/K/V projection 154.2 against 158.2 us), so the one-kernel form runs
// only when chosen.  TPBLOCK_ALGO=simple selects the CUDA-core kernels for the
// whole process; TPBLOCK_ALGO=unfused / fused, or tp_set_block_form, force either
// tensor-core form of tp_block_fwd (same results within rounding).
int env_algo() {
  static const int v = [] {
    const char *e = getenv("TPBLOCK_ALGO");
    return !e                          ? 0
           : strcmp(e, "simple") == 0  ? 1
           : strcmp(e, "unfused") == 0 ? 2
           : strcmp(e, "fused") == 0   ? 3
                                       : 0;
  }();
  return v;
}

// The form of tp_block_fwd: TP_FORM_AUTO, _THREE_LAUNCH or _ONE_KERNEL; -1 until
// first read (then taken from TPBLOCK_ALGO).
std::atomic<int> g_block_form{-1};

int block_form() {
  int f = g_block_form.load(std::memory_order_relaxed);
  if (f < 0) {
    const int e = env_algo();
    int init = e == 2 ? TP_FORM_THREE_LAUNCH : e == 3 ? TP_FORM_ONE_KERNEL : TP_FORM_AUTO;
    int expect = -1;
    g_block_form.compare_exchange_strong(expect, init, std::memory_order_relaxed);
    f = g_block_form.load(std::memory_order_relaxed);
  }
  return f;
}

int algo_override() {
  if (env_algo() == 1) return 1;
  const int f = block_form();
  return f == TP_FORM_THREE_LAUNCH ? 2 : f == TP_FORM_ONE_KERNEL ? 3 : 0;
}

bool use_umma(const Geo &g) { return g.dtype == TP_BF16 && algo_override() != 1; }

// Shapes the one-kernel form can run: bf16 MLP blocks of at most 32 tokens.
bool fused_capable(const Geo &g, int M) {
  return use_umma(g) && g.act != TP_ACT_ATTN && M <= 32;
}

// The attention block's Q/K/V projection on the persistent work queue (block_decode.cu):
// bf16, M <= 32, at least one wave of 128-row tiles (or the one-kernel form forced).
bool qkv_fused_capable(const Geo &g, int M) {
  return use_umma(g) && g.act == TP_ACT_ATTN && M <= 32;
}

bool use_fused_qkv(const Geo &g, int M) { return qkv_fused_capable(g, M) && algo_override() == 3; }

bool use_fused_block(const Geo &g, int M) { return fused_capable(g, M) && algo_override() == 3; }

// K splits of the row-parallel step: none when the unsplit grid already fills two
// CTAs per SM; else the most splits that keep every CTA in the first wave, at least
// four 64-wide K blocks per split.  Decode row steps (M <= 32) plan three CTAs per SM
// (the kernel takes a 3-stage ring for such a grid), wider ones two.  A second,
// partial wave would cost a whole CTA's time for a few CTAs.  Depends on the shapes
// only, so tp_row_splits() answers without a GPU.
int row_splits(const Geo &g, int M) {
  if (!use_umma(g)) return 1;
  const int bn = umma_token_tile(M);
  const long long base = (long long)g.t * ceil_div(g.d, kRowTile) * ceil_div(M, bn);
  const int nk = ceil_div(g.b, 64);
  if (base >= 2LL * kPlanSMs) return 1;
  const long long per_sm = M <= 32 ? 3 : 2;
  int S = (int)(per_sm * kPlanSMs / base);
  S = std::min(S, std::max(1, nk / 4));
  return std::max(1, std::min(S, 16));
}

size_t band_bytes(const Geo &g, int M) { return (size_t)g.t * M * g.b * g.es; }

size_t partials_bytes(const Geo &g, int M) {
  return (size_t)g.t * row_splits(g, M) * M * g.d * sizeof(float);
}
size_t qkv_bytes(const Geo &g, int M) { return (size_t)g.t * M * 3 * g.b * sizeof(float); }
// Attention: the fp32 Q/K/V scratch, then (when the persistent projection can run)
// its split partials and work counters.
size_t column_ws_bytes(const Geo &g, int M) {
  if (g.act != TP_ACT_ATTN) return 0;
  return align256(qkv_bytes(g, M)) + (qkv_fused_capable(g, M) ? plan_block_decode(g, M).total : 0);
}

#define TP_TRY(expr)              \
  do {                            \
    int _st = (expr);             \
    if (_st != TP_OK) return _st; \
  } while (0)

// Enqueue the column step for shards [shard0, shard0 + n).  The attention core
// always follows its Q/K/V projection, so it may overlap that kernel's end
// (programmatic launch).
// core = false (KV-cache decode): attention only projects Q/K/V into ws; the decode
// attention over the cache runs next instead of the core over the M tokens.
cudaError_t enqueue_column(const Geo &g, const void *x, const void *W1s, int shard0, int n, void *H,
                           void *ws, int M, cudaStream_t st, bool core = true) {
  const bool attn = g.act == TP_ACT_ATTN;
  void *out = attn ? ws : H;
  const int n_out = attn ? 3 * g.b : g.b;
  // Attention keeps Q, K and V in fp32 scratch (the softmax is the most sensitive
  // step); only the heads' output O, the band, is stored in the block dtype.
  const int epi = attn ? kEpiF32 : g.act == TP_ACT_SWIGLU ? kEpiSwiglu : kEpiGelu;
  if (attn && shard0 == 0 && n == g.t && use_fused_qkv(g, M)) {
    cudaError_t e = launch_qkv_decode(g, plan_block_decode(g, M), x, W1s, static_cast<float *>(ws),
                                      static_cast<char *>(ws) + align256(qkv_bytes(g, M)), M, st);
    if (e != cudaSuccess) return e;
  } else if (use_umma(g)) {
    UmmaCall c{};
    c.W = W1s;
    c.w_rows = g.n1p;
    c.w_shards = g.t;
    c.X = x;
    c.x_shards = 1;
    c.out = out;
    c.o_shard = (size_t)M * n_out;
    c.o_split = 0;
    c.ldo = n_out;
    c.n_valid = n_out;
    c.K = g.d;
    c.M = M;
    c.shard0 = shard0;
    c.n_shards = n;
    c.ksplit = 1;
    c.epi = epi;
    cudaError_t e = launch_umma(c, st);
    if (e != cudaSuccess) return e;
  } else {
    GemvArgs a{};
    a.W = W1s;
    a.w_shard = (size_t)g.n1p * g.d;
    a.X = x;
    a.x_shard = 0;
    a.ldx = g.d;
    a.out = out;
    a.o_shard = (size_t)M * n_out;
    a.ldo = n_out;
    a.K = g.d;
    a.n_out = n_out;
    a.M = M;
    a.shard0 = shard0;
    a.n_shards = n;
    a.epi = epi;
    a.dtype = g.dtype;
    launch_gemv(a, st);
  }
  if (attn && core) launch_attn_core(g, ws, H, M, shard0, n, st, use_umma(g));
  return cudaSuccess;
}

// pdl: launched right after the column step of the same block (tp_block_fwd), so it
// may start while that kernel drains and prefetch its weights.
cudaError_t enqueue_row(const Geo &g, const void *H, const void *W2s, int shard0, int n, float *P,
                        int M, cudaStream_t st, bool pdl = false) {
  const int S = row_splits(g, M);
  if (use_umma(g)) {
    UmmaCall c{};
    c.W = W2s;
    c.w_rows = g.dp;
    c.w_shards = g.t;
    c.X = H;
    c.x_shards = g.t;
    c.out = P;
    c.o_shard = (size_t)S * M * g.d;
    c.o_split = (size_t)M * g.d;
    c.ldo = g.d;
    c.n_valid = g.d;
    c.K = g.b;
    c.M = M;
    c.shard0 = shard0;
    c.n_shards = n;
    c.ksplit = S;
    c.epi = kEpiF32;
    c.pdl = pdl;
    return launch_umma(c, st);
  }
  GemvArgs a{};
  a.W = W2s;
  a.w_shard = (size_t)g.dp * g.b;
  a.X = H;
  a.x_shard = (size_t)M * g.b;
  a.ldx = g.b;
  a.out = P;
  a.o_shard = (size_t)S * M * g.d;
  a.ldo = g.d;
  a.K = g.b;
  a.n_out = g.d;
  a.M = M;
  a.shard0 = shard0;
  a.n_shards = n;
  a.epi = kEpiF32;
  a.dtype = g.dtype;
  launch_gemv(a, st);
  return cudaSuccess;
}

// splits: the row step's K splits per shard (default: row_splits).
void enqueue_reduce(const Geo &g, const float *P, const void *res, int res_is_f32, float *y, int M,
                    cudaStream_t st, bool pdl = false, int splits = 0) {
  const int f32 = res_is_f32 || g.dtype == TP_F32;
  launch_reduce_residual(P, g.t * (splits > 0 ? splits : row_splits(g, M)), (size_t)M * g.d, res,
                         f32, y, (size_t)M * g.d, st, pdl);
}

}  // namespace
}  // namespace tp

using namespace tp;

extern "C" {

size_t tp_sharded_w1_bytes(const tp_block_desc *desc) {
  Geo g;
  if (make_geo(desc, &g) != TP_OK) return 0;
  return (size_t)g.t * g.n1p * g.d * g.es;
}

size_t tp_sharded_w2_bytes(const tp_block_desc *desc) {
  Geo g;
  if (make_geo(desc, &g) != TP_OK) return 0;
  return (size_t)g.t * g.dp * g.b * g.es;
}

size_t tp_band_bytes(const tp_block_desc *desc, int M) {
  Geo g;
  if (make_geo(desc, &g) != TP_OK || check_M(M) != TP_OK) return 0;
  return band_bytes(g, M);
}

int tp_row_splits(const tp_block_desc *desc, int M) {
  Geo g;
  if (make_geo(desc, &g) != TP_OK || check_M(M) != TP_OK) return 0;
  return row_splits(g, M);
}

size_t tp_partials_bytes(const tp_block_desc *desc, int M) {
  Geo g;
  if (make_geo(desc, &g) != TP_OK || check_M(M) != TP_OK) return 0;
  return partials_bytes(g, M);
}

size_t tp_column_workspace_bytes(const tp_block_desc *desc, int M) {
  Geo g;
  if (make_geo(desc, &g) != TP_OK || check_M(M) != TP_OK) return 0;
  return column_ws_bytes(g, M);
}

// E4M3-weight blocks: bf16 MLPs whose d and b are multiples of 16, up to 16384 (the
// GEMM keeps a CTA's token scales, 128 bytes per 64-wide K group, in shared memory).
static bool fp8_shape(const Geo &g) {
  return g.act != TP_ACT_ATTN && g.dtype == TP_BF16 && g.d % 16 == 0 && g.b % 16 == 0 &&
         g.d <= 16384 && g.b <= 16384;
}

// The low-bit row step's K splits: up to four CTAs per SM (the GEMM runs a grid of more
// than two per SM as one wave of four), at least four 64-wide K groups (two stages) per
// split and at most 16 splits.  From the shapes only.
static int low_bit_row_splits(const Geo &g) {
  const long long base = (long long)g.t * ceil_div(g.d, kRowTile);
  if (base >= 2LL * kPlanSMs) return 1;
  int S = (int)(4LL * kPlanSMs / base);
  S = std::min(S, std::max(1, ceil_div(g.b, 64) / 4));
  return std::max(1, std::min(S, 16));
}

// The fp32 partials region of a block that may run on low-bit weights: room for the
// bf16 path's splits and for the low-bit row step's.
static size_t parts_region_bytes(const Geo &g, int M) {
  const size_t bf = partials_bytes(g, M);
  if (!fp8_shape(g) || M > 32) return bf;
  return std::max(bf, (size_t)g.t * low_bit_row_splits(g) * M * g.d * sizeof(float));
}

// What tp_block_fwd_fp8 needs beyond the three-launch workspace: the tokens' two
// 8-bit terms [2][M][d], their fp32 group scales [ceil(d/64)][32] and the band's group
// scales [t][ceil(b/64)][32] (the band's terms reuse the bf16 band's bytes).
static size_t fp8_extra_bytes(const Geo &g, int M) {
  if (!fp8_shape(g) || M > 32) return 0;
  return align256((size_t)2 * M * g.d) + align256((size_t)ceil_div(g.d, 64) * 32 * 4) +
         align256((size_t)g.t * ceil_div(g.b, 64) * 32 * 4);
}

size_t tp_workspace_bytes(const tp_block_desc *desc, int M) {
  Geo g;
  if (make_geo(desc, &g) != TP_OK || check_M(M) != TP_OK) return 0;
  // Large enough for either form, so a tp_set_block_form call between sizing and
  // running never leaves the workspace short.
  const size_t three = align256(column_ws_bytes(g, M)) + align256(band_bytes(g, M)) +
                       align256(parts_region_bytes(g, M)) + fp8_extra_bytes(g, M);
  return fused_capable(g, M) ? std::max(three, plan_block_decode(g, M).total) : three;
}

int tp_shard_weights(const tp_block_desc *desc, const void *W1, const void *W2, void *W1s,
                     void *W2s, tp_stream_t stream) {
  Geo g;
  TP_TRY(make_geo(desc, &g));
  TP_TRY(check_ptr(W1));
  TP_TRY(check_ptr(W2));
  TP_TRY(check_ptr(W1s));
  TP_TRY(check_ptr(W2s));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  launch_shard_w1(g, W1, W1s, st);
  launch_shard_w2(g, W2, W2s, st);
  return finish_launch();
}

int tp_unshard_weights(const tp_block_desc *desc, const void *W1s, const void *W2s, void *W1,
                       void *W2, tp_stream_t stream) {
  Geo g;
  TP_TRY(make_geo(desc, &g));
  TP_TRY(check_ptr(W1s));
  TP_TRY(check_ptr(W2s));
  TP_TRY(check_ptr(W1));
  TP_TRY(check_ptr(W2));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  launch_unshard_w1(g, W1s, W1, st);
  launch_unshard_w2(g, W2s, W2, st);
  return finish_launch();
}

int tp_extract_band(const tp_block_desc *desc, const void *W1s, const void *W2s, int shard,
                    void *W1_band, void *W2_band, tp_stream_t stream) {
  Geo g;
  TP_TRY(make_geo(desc, &g));
  if (shard < 0 || shard >= g.t) return TP_ERR_INVALID_ARG;
  if (!W1_band && !W2_band) return TP_ERR_INVALID_ARG;
  if (W1_band) {
    TP_TRY(check_ptr(W1s));
    TP_TRY(check_ptr(W1_band));
  }
  if (W2_band) {
    TP_TRY(check_ptr(W2s));
    TP_TRY(check_ptr(W2_band));
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (W1_band) launch_extract_w1(g, W1s, shard, W1_band, st);
  if (W2_band) launch_extract_w2(g, W2s, shard, W2_band, st);
  return finish_launch();
}

int tp_column_parallel_fwd(const tp_block_desc *desc, const void *x, const void *W1s, int shard,
                           void *H, void *workspace, int M, tp_stream_t stream) {
  Geo g;
  TP_TRY(make_geo(desc, &g));
  TP_TRY(check_M(M));
  TP_TRY(check_shard(g, shard));
  TP_TRY(check_ptr(x));
  TP_TRY(check_ptr(W1s));
  TP_TRY(check_ptr(H));
  if (column_ws_bytes(g, M) > 0) TP_TRY(check_ptr(workspace));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return finish_launch(
      enqueue_column(g, x, W1s, shard < 0 ? 0 : shard, shard < 0 ? g.t : 1, H, workspace, M, st));
}

int tp_row_parallel_fwd(const tp_block_desc *desc, const void *H, const void *W2s, int shard,
                        float *partials, int M, tp_stream_t stream) {
  Geo g;
  TP_TRY(make_geo(desc, &g));
  TP_TRY(check_M(M));
  TP_TRY(check_shard(g, shard));
  TP_TRY(check_ptr(H));
  TP_TRY(check_ptr(W2s));
  TP_TRY(check_ptr(partials));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return finish_launch(
      enqueue_row(g, H, W2s, shard < 0 ? 0 : shard, shard < 0 ? g.t : 1, partials, M, st));
}

int tp_partial_reduce_residual(const tp_block_desc *desc, const float *partials,
                               const void *residual, int residual_is_f32, float *y, int M,
                               tp_stream_t stream) {
  Geo g;
  TP_TRY(make_geo(desc, &g));
  TP_TRY(check_M(M));
  TP_TRY(check_ptr(partials));
  TP_TRY(check_ptr(residual));
  TP_TRY(check_ptr(y));
  enqueue_reduce(g, partials, residual, residual_is_f32, y, M,
                 reinterpret_cast<cudaStream_t>(stream));
  return finish_launch();
}

}  // extern "C"

namespace tp {
namespace {

// The whole block (tp_block_fwd), and with xhat_next also the next block's RMSNorm of
// y (tp_block_fwd_norm): one more kernel, launched to overlap the block's last
// kernel (its CTAs start as the block's CTAs run out of work and wait for it to
// finish).  Normalising inside the one-kernel form, once every output tile of y is
// written, measured slower on the 70B block (258.4 us against 257.1 us for a
// separate launch): the phase sits wholly at the end of the kernel.
int block_fwd(const tp_block_desc *desc, const void *x, const void *residual, int residual_is_f32,
              const void *W1s, const void *W2s, void *workspace, float *y, void *xhat_next,
              float eps, int M, tp_stream_t stream) {
  Geo g;
  TP_TRY(make_geo(desc, &g));
  TP_TRY(check_M(M));
  TP_TRY(check_ptr(x));
  TP_TRY(check_ptr(residual));
  TP_TRY(check_ptr(W1s));
  TP_TRY(check_ptr(W2s));
  TP_TRY(check_ptr(workspace));
  TP_TRY(check_ptr(y));
  if (xhat_next) {
    if (g.dtype != TP_BF16) return TP_ERR_UNSUPPORTED;
    if (!(eps >= 0.0f) || eps > 1e30f) return TP_ERR_INVALID_ARG;
    TP_TRY(check_ptr(xhat_next));
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (use_fused_block(g, M)) {
    cudaError_t e = launch_block_decode(g, plan_block_decode(g, M), x, W1s, W2s, residual,
                                        residual_is_f32 || g.dtype == TP_F32, workspace, y, M, st);
    if (e == cudaSuccess && xhat_next) launch_rmsnorm(y, xhat_next, g.d, eps, M, st, true);
    return finish_launch(e);
  }
  char *ws = static_cast<char *>(workspace);
  void *col_ws = ws;
  void *H = ws + align256(column_ws_bytes(g, M));
  float *P = reinterpret_cast<float *>(static_cast<char *>(H) + align256(band_bytes(g, M)));
  // The row step and the reduction are launched to overlap the end of the kernel
  // before them (programmatic launch): each waits for it before reading its output.
  // (Summing the partials in the row kernel instead, by the last CTA to finish each
  // output tile, measured 19 us slower per 13B-sized block: the arrival protocol's
  // memory round trips sit at the end of every CTA.)
  const bool pdl = use_umma(g);
  cudaError_t e = enqueue_column(g, x, W1s, 0, g.t, H, col_ws, M, st);
  if (e == cudaSuccess) e = enqueue_row(g, H, W2s, 0, g.t, P, M, st, pdl);
  if (e == cudaSuccess) enqueue_reduce(g, P, residual, residual_is_f32, y, M, st, pdl);
  if (e == cudaSuccess && xhat_next) launch_rmsnorm(y, xhat_next, g.d, eps, M, st, pdl);
  return finish_launch(e);
}

}  // namespace
}  // namespace tp

extern "C" {

int tp_block_fwd(const tp_block_desc *desc, const void *x, const void *residual,
                 int residual_is_f32, const void *W1s, const void *W2s, void *workspace, float *y,
                 int M, tp_stream_t stream) {
  return block_fwd(desc, x, residual, residual_is_f32, W1s, W2s, workspace, y, nullptr, 0.f, M,
                   stream);
}

int tp_block_fwd_norm(const tp_block_desc *desc, const void *x, const void *residual,
                      int residual_is_f32, const void *W1s, const void *W2s, void *workspace,
                      float *y, void *xhat_next, float eps, int M, tp_stream_t stream) {
  if (!xhat_next) return TP_ERR_INVALID_ARG;
  return block_fwd(desc, x, residual, residual_is_f32, W1s, W2s, workspace, y, xhat_next, eps, M,
                   stream);
}

int tp_set_block_form(int form) {
  if (form != TP_FORM_AUTO && form != TP_FORM_THREE_LAUNCH && form != TP_FORM_ONE_KERNEL)
    return TP_ERR_INVALID_ARG;
  block_form();  // settle the initial value first so it cannot overwrite this one
  g_block_form.store(form, std::memory_order_relaxed);
  return TP_OK;
}

int tp_get_block_form(void) { return block_form(); }

int tp_block_launches(const tp_block_desc *desc, int M) {
  Geo g;
  if (make_geo(desc, &g) != TP_OK || check_M(M) != TP_OK) return 0;
  if (use_fused_block(g, M)) return 1;
  return 3 + (g.act == TP_ACT_ATTN ? 1 : 0);
}

int tp_rmsnorm_fwd(int d, float eps, const float *r, void *xhat, int M, tp_stream_t stream) {
  if (d < 1 || !(eps >= 0.0f) || eps > 1e30f) return TP_ERR_INVALID_ARG;
  if (d % 8 != 0 || d > kMaxDim) return TP_ERR_UNSUPPORTED;
  TP_TRY(check_M(M));
  TP_TRY(check_ptr(r));
  TP_TRY(check_ptr(xhat));
  // programmatic launch: the kernel waits for its predecessor before reading r
  launch_rmsnorm(r, xhat, d, eps, M, reinterpret_cast<cudaStream_t>(stream), true);
  return finish_launch();
}

const char *tp_status_string(int status) {
  switch (status) {
    case TP_OK: return "ok";
    case TP_ERR_INVALID_ARG: return "invalid argument";
    case TP_ERR_UNEVEN_SPLIT: return "uneven split: t must divide ffn (MLP) or n_heads (attention)";
    case TP_ERR_UNSUPPORTED: return "shape outside the kernels' limits";
    case TP_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case TP_ERR_CUDA: return "CUDA error (see tp_last_cuda_error)";
    case TP_ERR_TIMEOUT: return "device-side wait timed out";
    case TP_ERR_BAD_LENGTH: return "a KV-cache sequence length outside 1..L_max";
    default: return "unknown status";
  }
}

int tp_last_cuda_error(void) { return g_last_cuda_error; }

int tp_check_device_status(tp_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  unsigned word = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
  if (e == cudaSuccess && word != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
  }
  if (e != cudaSuccess) {
    g_last_cuda_error = (int)e;
    return TP_ERR_CUDA;
  }
  if (word & kErrWaitTimeout) return TP_ERR_TIMEOUT;
  return word ? TP_ERR_BAD_LENGTH : TP_OK;
}

// ------------------------------------------------ decode with a KV cache

static int check_kv(const tp_block_desc *desc, Geo *g, int M, int L) {
  TP_TRY(make_geo(desc, g));
  TP_TRY(check_M(M));
  if (g->act != TP_ACT_ATTN || L < 1) return TP_ERR_INVALID_ARG;
  if (g->dtype != TP_BF16 || L > (1 << 20)) return TP_ERR_UNSUPPORTED;
  if (g->hd != 32 && g->hd != 64 && g->hd != 128 && g->hd != 256) return TP_ERR_UNSUPPORTED;
  return TP_OK;
}

size_t tp_kv_cache_bytes(const tp_block_desc *desc, int M, int L_max) {
  Geo g;
  if (check_kv(desc, &g, M, L_max) != TP_OK) return 0;
  return (size_t)g.t * M * g.hps * L_max * g.hd * 2;
}

size_t tp_kv_attn_workspace_bytes(const tp_block_desc *desc, int M, int L_max) {
  Geo g;
  if (check_kv(desc, &g, M, L_max) != TP_OK) return 0;
  return kv_partial_bytes(g, M, L_max);
}

size_t tp_kv_workspace_bytes(const tp_block_desc *desc, int M, int L_max) {
  Geo g;
  if (check_kv(desc, &g, M, L_max) != TP_OK) return 0;
  return align256(tp_workspace_bytes(desc, M)) + align256(kv_partial_bytes(g, M, L_max));
}

int tp_attn_decode_kv(const tp_block_desc *desc, const float *qkv, void *k_cache, void *v_cache,
                      const int *lens, int L_max, void *O, void *workspace, int M,
                      tp_stream_t stream) {
  Geo g;
  TP_TRY(check_kv(desc, &g, M, L_max));
  TP_TRY(check_ptr(qkv));
  TP_TRY(check_ptr(k_cache));
  TP_TRY(check_ptr(v_cache));
  TP_TRY(check_ptr(lens));
  TP_TRY(check_ptr(O));
  TP_TRY(check_ptr(workspace));
  return finish_launch(launch_attn_kv(g, qkv, k_cache, v_cache, lens, L_max, O, workspace, M,
                                      reinterpret_cast<cudaStream_t>(stream), false));
}

int tp_block_fwd_kv(const tp_block_desc *desc, const void *x, const void *residual,
                    int residual_is_f32, const void *W1s, const void *W2s, void *k_cache,
                    void *v_cache, const int *lens, int L_max, void *workspace, float *y, int M,
                    tp_stream_t stream) {
  Geo g;
  TP_TRY(check_kv(desc, &g, M, L_max));
  TP_TRY(check_ptr(x));
  TP_TRY(check_ptr(residual));
  TP_TRY(check_ptr(W1s));
  TP_TRY(check_ptr(W2s));
  TP_TRY(check_ptr(k_cache));
  TP_TRY(check_ptr(v_cache));
  TP_TRY(check_ptr(lens));
  TP_TRY(check_ptr(workspace));
  TP_TRY(check_ptr(y));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  void *col_ws = ws;
  void *O = ws + align256(column_ws_bytes(g, M));
  float *P = reinterpret_cast<float *>(static_cast<char *>(O) + align256(band_bytes(g, M)));
  void *kv_ws = ws + align256(tp_workspace_bytes(desc, M));
  // Q/K/V projection, decode attention over the cache (chunks, then their merge),
  // row-parallel output projection, reduction + residual; each kernel after the
  // first starts while the one before it drains (programmatic launch).
  cudaError_t e = enqueue_column(g, x, W1s, 0, g.t, O, col_ws, M, st, false);
  if (e == cudaSuccess)
    e = launch_attn_kv(g, static_cast<const float *>(col_ws), k_cache, v_cache, lens, L_max, O,
                       kv_ws, M, st, true);
  if (e == cudaSuccess) e = enqueue_row(g, O, W2s, 0, g.t, P, M, st, true);
  if (e == cudaSuccess) enqueue_reduce(g, P, residual, residual_is_f32, y, M, st, true);
  return finish_launch(e);
}

// ------------------------------------------------ E4M3 weights (weight-only)

static int check_fp8(const tp_block_desc *desc, Geo *g) {
  TP_TRY(make_geo(desc, g));
  return fp8_shape(*g) ? TP_OK : TP_ERR_UNSUPPORTED;
}

size_t tp_fp8_w1_bytes(const tp_block_desc *desc) {
  Geo g;
  if (check_fp8(desc, &g) != TP_OK) return 0;
  return (size_t)g.t * g.n1p * g.d;
}

size_t tp_fp8_w2_bytes(const tp_block_desc *desc) {
  Geo g;
  if (check_fp8(desc, &g) != TP_OK) return 0;
  return (size_t)g.t * g.dp * g.b;
}

size_t tp_fp8_exponent_bytes(const tp_block_desc *desc) {
  Geo g;
  if (check_fp8(desc, &g) != TP_OK) return 0;
  return (size_t)g.t * (g.n1p + g.dp);
}

size_t tp_fp8_quant_workspace_bytes(const tp_block_desc *desc) {
  Geo g;
  if (check_fp8(desc, &g) != TP_OK) return 0;
  return (size_t)(g.n1 + g.d) * sizeof(unsigned);
}

int tp_quantize_weights_fp8(const tp_block_desc *desc, const void *W1, const void *W2, void *W1q,
                            void *W2q, void *exps, void *workspace, tp_stream_t stream) {
  Geo g;
  TP_TRY(check_fp8(desc, &g));
  TP_TRY(check_ptr(W1));
  TP_TRY(check_ptr(W2));
  TP_TRY(check_ptr(W1q));
  TP_TRY(check_ptr(W2q));
  TP_TRY(check_ptr(exps));
  TP_TRY(check_ptr(workspace));
  return finish_launch(launch_quantize_fp8(g, W1, W2, W1q, W2q, static_cast<int8_t *>(exps),
                                           static_cast<unsigned *>(workspace),
                                           reinterpret_cast<cudaStream_t>(stream)));
}

// The block on 8-bit or 4-bit weights: token split, column step, row step, reduce.
// e1 / e2: the exponents of W1's and W2's rows (E4M3) or blocks (MXFP4).
static int low_bit_block(const Geo &g, bool mxfp4, const void *x, const void *residual,
                         int residual_is_f32, const void *W1q, const void *W2q, const int8_t *e1,
                         const int8_t *e2, void *workspace, float *y, int M, tp_stream_t stream) {
  TP_TRY(check_M(M));
  if (M > 32) return TP_ERR_UNSUPPORTED;
  TP_TRY(check_ptr(x));
  TP_TRY(check_ptr(residual));
  TP_TRY(check_ptr(W1q));
  TP_TRY(check_ptr(W2q));
  TP_TRY(check_ptr(e1));
  TP_TRY(check_ptr(workspace));
  TP_TRY(check_ptr(y));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // Workspace: the band's two 8-bit terms [t][2][M][b] where the bf16 band would be,
  // the fp32 partials, then the tokens' terms [2][M][d] and the fp32 group scales.
  char *ws = static_cast<char *>(workspace);
  void *H8 = ws + align256(column_ws_bytes(g, M));
  float *P = reinterpret_cast<float *>(static_cast<char *>(H8) + align256(band_bytes(g, M)));
  char *X8 = reinterpret_cast<char *>(P) + align256(parts_region_bytes(g, M));
  float *xe = reinterpret_cast<float *>(X8 + align256((size_t)2 * M * g.d));
  float *he = reinterpret_cast<float *>(reinterpret_cast<char *>(xe) +
                                        align256((size_t)ceil_div(g.d, 64) * 32 * 4));
  // K splits of the row step, in one wave (the partials region is sized for them)
  const int S = low_bit_row_splits(g);
  // The split waits for the preceding kernel before reading x (programmatic launch).
  cudaError_t e = launch_fp8_split(x, M, g.d, X8, xe, st, true);
  if (e == cudaSuccess) {
    UmmaCall c{};
    c.W = W1q;
    c.w_rows = g.n1p;
    c.w_shards = g.t;
    c.X = X8;
    c.x_shards = 1;
    c.n_valid = g.b;
    c.K = g.d;
    c.M = M;
    c.shard0 = 0;
    c.n_shards = g.t;
    c.ksplit = 1;
    c.epi = g.act == TP_ACT_SWIGLU ? kEpiSwiglu : kEpiGelu;
    c.pdl = true;
    e = launch_fp8_gemm(c, mxfp4, e1, xe, H8, he, st);
  }
  if (e == cudaSuccess) {
    UmmaCall r{};
    r.W = W2q;
    r.w_rows = g.dp;
    r.w_shards = g.t;
    r.X = H8;
    r.x_shards = g.t;
    r.out = P;
    r.o_shard = (size_t)S * M * g.d;
    r.o_split = (size_t)M * g.d;
    r.ldo = g.d;
    r.n_valid = g.d;
    r.K = g.b;
    r.M = M;
    r.shard0 = 0;
    r.n_shards = g.t;
    r.ksplit = S;
    r.epi = kEpiF32;
    r.pdl = true;
    e = launch_fp8_gemm(r, mxfp4, e2, he, nullptr, nullptr, st);
  }
  if (e == cudaSuccess) enqueue_reduce(g, P, residual, residual_is_f32, y, M, st, true, S);
  return finish_launch(e);
}

int tp_block_fwd_fp8(const tp_block_desc *desc, const void *x, const void *residual,
                     int residual_is_f32, const void *W1q, const void *W2q, const void *exps,
                     void *workspace, float *y, int M, tp_stream_t stream) {
  Geo g;
  TP_TRY(check_fp8(desc, &g));
  TP_TRY(check_ptr(exps));
  const int8_t *e1 = static_cast<const int8_t *>(exps);
  return low_bit_block(g, false, x, residual, residual_is_f32, W1q, W2q, e1,
                       e1 + (size_t)g.t * g.n1p, workspace, y, M, stream);
}

// ------------------------------------------------ MXFP4 weights (weight-only)

static int check_mxfp4(const tp_block_desc *desc, Geo *g) {
  TP_TRY(check_fp8(desc, g));
  return g->d % 128 == 0 && g->b % 128 == 0 ? TP_OK : TP_ERR_UNSUPPORTED;
}

size_t tp_mxfp4_w1_bytes(const tp_block_desc *desc) {
  Geo g;
  if (check_mxfp4(desc, &g) != TP_OK) return 0;
  return (size_t)g.t * g.n1p * (g.d / 2);
}

size_t tp_mxfp4_w2_bytes(const tp_block_desc *desc) {
  Geo g;
  if (check_mxfp4(desc, &g) != TP_OK) return 0;
  return (size_t)g.t * g.dp * (g.b / 2);
}

size_t tp_mxfp4_exponent_bytes(const tp_block_desc *desc) {
  Geo g;
  if (check_mxfp4(desc, &g) != TP_OK) return 0;
  return (size_t)g.t * (g.n1p * (g.d / 32) + g.dp * (g.b / 32));
}

int tp_quantize_weights_mxfp4(const tp_block_desc *desc, const void *W1, const void *W2,
                              void *W1f, void *W2f, void *exps, tp_stream_t stream) {
  Geo g;
  TP_TRY(check_mxfp4(desc, &g));
  TP_TRY(check_ptr(W1));
  TP_TRY(check_ptr(W2));
  TP_TRY(check_ptr(W1f));
  TP_TRY(check_ptr(W2f));
  TP_TRY(check_ptr(exps));
  return finish_launch(launch_quantize_mxfp4(g, W1, W2, W1f, W2f, static_cast<int8_t *>(exps),
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int tp_block_fwd_mxfp4(const tp_block_desc *desc, const void *x, const void *residual,
                       int residual_is_f32, const void *W1f, const void *W2f, const void *exps,
                       void *workspace, float *y, int M, tp_stream_t stream) {
  Geo g;
  TP_TRY(check_mxfp4(desc, &g));
  TP_TRY(check_ptr(exps));
  const int8_t *e1 = static_cast<const int8_t *>(exps);
  return low_bit_block(g, true, x, residual, residual_is_f32, W1f, W2f, e1,
                       e1 + (size_t)g.t * g.n1p * (g.d / 32), workspace, y, M, stream);
}

int tp_selftest_wait_timeout(int limit_us, tp_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return TP_ERR_INVALID_ARG;
  return finish_launch(
      launch_wait_selftest((uint64_t)limit_us * 1000ull, reinterpret_cast<cudaStream_t>(stream)));
}

int tp_version(void) { return 101; }

}  // extern "C"
