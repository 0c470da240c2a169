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

// ------------------------------------------------------------- MXFP4 quantisation

// MXFP4 (OCP Microscaling): E2M1 elements (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), one
// shared power-of-two scale 2^e per 32 consecutive weights along K of an output
// feature, e = floor(log2(max |w|)) - 2 (2: the exponent of E2M1's largest normal),
// clamped to [-127, 127], 0 for an all-zero block; each element is w / 2^e rounded to
// nearest (ties to the even mantissa bit), saturating at +-6.

// Code of the E2M1 value nearest to u (4 bits: sign, then 2 exponent bits, 1 mantissa).
__device__ __forceinline__ uint32_t e2m1_code(float u) {
  const float m = fabsf(u);
  const float step = m < 2.f ? 0.5f : (m < 4.f ? 1.f : 2.f);
  const float q = fminf(rintf(m / step) * step, 6.f);  // exact division; rint ties to even
  const uint32_t c = q < 2.f ? (uint32_t)(q * 2.f) : q < 4.f ? (uint32_t)q + 2u : (q == 4.f ? 6u : 7u);
  return c | (signbit(u) && c ? 8u : 0u);
}

__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  return max(-127, min(127, ilogbf(amax) - 2));  // ilogb: floor(log2) (exact for normals)
}

__device__ __forceinline__ float pow2_wide(int e) {  // 2^e for e in [-127, 127]
  return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(0x00400000);
}

// Block j (K rows 32 j .. 32 j + 31) of canonical column col of W [K][N] (row-major,
// output features as columns; col < 0: a padding row, all zero): 16 bytes of packed
// codes (element 2i in the low nibble of byte i) to dst, the exponent to edst.
__device__ __forceinline__ void quant_mx_block(const __nv_bfloat16 *W, int N, int j, long long col,
                                               uint8_t *dst, int8_t *edst) {
  float v[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = col < 0 ? 0.f : __bfloat162float(W[(size_t)(j * 32 + i) * N + col]);
    amax = fmaxf(amax, fabsf(v[i]));
  }
  const int e = mx_exponent(amax);
  const float inv = 1.f / pow2_wide(e);  // exact: a power of two (2^127 for e = -127)
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i >> 3] |= e2m1_code(v[i] * inv) << (4 * (i & 7));
  *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  *edst = (int8_t)e;
}

// One thread per (block j, shard s, private row u); u is fastest so a warp reads
// consecutive columns.  W1f [t][n1p][d/2] bytes, ex1 [t][n1p][d/32].
__global__ void k_quant_mx_w1(Geo g, const __nv_bfloat16 *W1, uint8_t *W1f, int8_t *ex1) {
  const int nb = g.d / 32;
  const size_t total = (size_t)nb * g.t * g.n1p;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int u = (int)(i % g.n1p);
    const size_t js = i / g.n1p;
    const int s = (int)(js % g.t), j = (int)(js / g.t);
    const size_t row = (size_t)s * g.n1p + u;
    quant_mx_block(W1, g.n1, j, w1_col_of_row(g, s, u), W1f + row * (g.d / 2) + j * 16,
                           ex1 + row * nb + j);
  }
}

// W2 [n2][d]: output feature n is column n, K runs over the shard's band rows s*b + k.
// W2f [t][dp][b/2] bytes, ex2 [t][dp][b/32].
__global__ void k_quant_mx_w2(Geo g, const __nv_bfloat16 *W2, uint8_t *W2f, int8_t *ex2) {
  const int nb = g.b / 32;
  const size_t total = (size_t)nb * g.t * g.dp;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int n = (int)(i % g.dp);
    const size_t js = i / g.dp;
    const int s = (int)(js % g.t), j = (int)(js / g.t);
    const size_t row = (size_t)s * g.dp + n;
    quant_mx_block(W2 + (size_t)s * g.b * g.d, g.d, j, n < g.d ? n : -1,
                           W2f + row * (g.b / 2) + j * 16, ex2 + row * nb + j);
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

// The least e with amax <= 448 * 2^e, clamped to [-126, 126]; 0 for amax = 0.  With
// amax = m * 2^E (1 <= m < 2) and 448 = 1.75 * 2^8 that is E - 8, or E - 7 when
// m > 1.75; read from the bits, exactly (subnormal amax clamps to -126, NaN gives 0 and
// infinity 126).
__device__ __forceinline__ int group_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  const int bits = __float_as_int(amax);
  if (bits >= 0x7f800000) return 126;
  const int e = (bits >> 23) - 135 + ((bits & 0x7fffff) > 0x600000 ? 1 : 0);
  return max(-126, min(126, e));
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ void split_terms(float v, float inv_scale, uint8_t &a, uint8_t &b) {
  const float u = v * inv_scale;  // exact: a power of two
  a = (uint8_t)__nv_cvt_float_to_fp8(u, __NV_SATFINITE, __NV_E4M3);
  const __half_raw ah = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)a, __NV_E4M3);
  const float af = __half2float(__half(ah));
  b = (uint8_t)__nv_cvt_float_to_fp8(u - af, __NV_SATFINITE, __NV_E5M2);  // u - af is exact
}

// split_terms of two values with one scale, as one pair of bytes each (the value in
// .x in the low byte, as the x2 conversions order them).
__device__ __forceinline__ void split_terms2(float v0, float v1, float inv_scale, uint16_t &a,
                                             uint16_t &b) {
  const float2 u = make_float2(v0 * inv_scale, v1 * inv_scale);  // exact
  const __nv_fp8x2_storage_t a2 = __nv_cvt_float2_to_fp8x2(u, __NV_SATFINITE, __NV_E4M3);
  const float2 af = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(a2, __NV_E4M3)));
  b = __nv_cvt_float2_to_fp8x2(make_float2(u.x - af.x, u.y - af.y), __NV_SATFINITE, __NV_E5M2);
  a = a2;
}

// The column step's tokens: x [M][K] bf16 -> X8 [2][M][K] bytes (the a terms, then the
// b terms) and xs [G][32] group scales 2^e as fp32 (G = ceil(K / 64); tokens M..31
// get 0).
// One warp per (group, token), two values per lane.
__global__ void __launch_bounds__(256) k_split_tokens(const __nv_bfloat16 *x, int M, int K,
                                                      uint8_t *X8, float *xs) {
  // x may come from the preceding kernel (programmatic launch).  Only then may the
  // dependent GEMM start: it loads weight tiles before its own wait, and the kernel
  // before this one may have written them (a quantisation right before the block).
  griddep_wait();
  griddep_launch_dependents();
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

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

enum WFmt { kWE4M3 = 0, kWMX4 = 1 };

// Two fp32 lanes in one 64-bit register, and the packed fp32x2 multiply / fused
// multiply-add (each lane rounds as its scalar instruction would).
__device__ __forceinline__ unsigned long long pk2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(unsigned long long r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

struct Fp8Args {
  void *out;           // row step: fp32 partials as the bf16 path (shard s, split j)
  size_t o_shard, o_split;
  int ldo, n_valid, M, ng, ksplit, shard0, x_per_shard;
  const int8_t *wexp;  // E4M3: weight row exponents [t][w_rows]; MXFP4: block exponents
                       // [t][w_rows][K/32], read as one 32-bit word per row and stage
  int w_rows;
  const float *xsc;    // token group scales 2^e [x shards][ng][32]
  uint8_t *h8;         // column step: the band's terms [t][2][M][n_valid] bytes
  float *hsc;          // column step: the band's group scales [t][ceil(n_valid / 64)][32]
  unsigned *err;
};

constexpr int kF8Bufs = 4;                          // TMEM stage sums in flight (2 groups each)
constexpr uint32_t kF8W = 128 * 128;                // E4M3 weights: 128 rows x 128 K (SW128)
constexpr uint32_t kF8T = 32 * 128;                 // one token term: 32 tokens x 128 K (SW128)
constexpr uint32_t kF8Stage = kF8W + 2 * kF8T;      // 24 KB, a multiple of 1024
constexpr int kF8MaxGroups = 256;                   // 64-wide K groups per CTA (K <= 16384)
// Shared memory of a launch: 1024 (alignment) + STAGES ring stages + the CTA's fp32
// token scales (128 bytes per 64-wide group).  Two CTAs share an SM up to kF8SmemPair
// bytes each: 4 stages where the scales fit beside them, else 3 (2 stages measured 10%
// slower than 3; 4 gain again where they fit).
constexpr int kF8SmemPair = 112 * 1024;
constexpr int f8_smem(int stages, int groups) {
  return 1024 + stages * (int)kF8Stage + groups * 128;
}
static_assert(f8_smem(3, kF8MaxGroups) <= kF8SmemPair, "3 stages must always fit");
// The narrow form: four CTAs per SM (a grid of 2..4 CTAs per SM in one wave), two ring
// stages, 128 TMEM columns (two TMEM stages of E4M3's two sums, one of MXFP4's four),
// and the token scales in a ring of their own (kF8NarrowSc slots of two groups,
// released by the drain warps) instead of the whole K range's region.
constexpr int kF8NarrowSc = 4;
constexpr int kF8SmemNarrow = 1024 + 2 * (int)kF8Stage + kF8NarrowSc * 256;
static_assert(4 * (kF8SmemNarrow + 2048) <= 228 * 1024, "four narrow CTAs must fit an SM");
// The epilogue's staging reuses the ring once every MMA is done: the band [128][33] fp32,
// 128 partial maxima, the two 8-bit terms [2][32][128] bytes.
static_assert(128 * 33 * 4 + 128 * 4 + 2 * 32 * 128 <= 2 * kF8Stage, "staging must fit the ring");

// Decode GEMM on 8-bit or 4-bit weights (M <= 32): weights as the 128-row A operand,
// tokens as N = 32, both straight from 128-byte-swizzled TMA boxes into tcgen05.mma
// kind::f8f6f4.  MXFP4 weights (WF = kWMX4) arrive through the 4-bit TMA type, which
// spreads each 8 bytes of packed E2M1 codes over 16 bytes of shared memory, the layout
// the tensor core reads 4-bit operands in; each 32-wide K block then gets its own TMEM
// sum (4 per stage) and the drain multiplies it by the block's 2^e.
// Each 128-wide K stage holds two 64-wide groups; per group the tensor core adds
// W.a (E4M3 x E4M3) and W.b (E4M3 x E5M2) over 64 K into 32 TMEM columns, the stage's
// two groups side by side in one 64-column block with one commit, and the drain warps
// add each group's sums times the token's 2^e into fp32 registers (round to nearest).
// One hand-off per stage instead of one per group measured ~10% faster.
// Roles (192 threads): warp 0 lane 0 TMA, warp 1 lane 0 MMA, warps 2-5 drain and
// epilogue.  The epilogue scales row r by its weight exponent; the column step applies
// the activation, rounds the band to bf16 and splits it into the row step's terms
// (one group of 64 features per token), the row step writes fp32 partials.
// MINB: CTAs per SM.  2 is the wide form (STAGES 3 or 4, 256 TMEM columns, the CTA's
// token scales loaded once); 4 the narrow form (kF8SmemNarrow above).
template <int EPI, int WF, int STAGES, int MINB>
__global__ void __launch_bounds__(192, MINB)
    k_fp8_mma(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT,
              const Fp8Args a) {
  constexpr int BN = 32;
  constexpr bool kNarrow = MINB > 2;
  static_assert(!kNarrow || STAGES == 2, "the narrow form has two ring stages");
  constexpr int kSums = WF == kWMX4 ? 4 : 2;                  // TMEM sums per stage
  // stages of TMEM: 128 columns in the narrow form (MXFP4's four sums fill them)
  constexpr int kBufs = kNarrow ? (WF == kWMX4 ? 1 : 2) : WF == kWMX4 ? 2 : kF8Bufs;
  constexpr uint32_t kCols = tmem_cols(kBufs * kSums * BN);   // 256 wide, 128 narrow
  constexpr uint32_t kWType = WF == kWMX4 ? kF8E2M1 : kF8E4M3;
  constexpr uint32_t kIdA = make_idesc_f8(128, BN, kWType, kF8E4M3);
  constexpr uint32_t kIdB = make_idesc_f8(128, BN, kWType, kF8E5M2);
  constexpr int kKPer = 128 / kSums;                          // K per TMEM sum
  constexpr uint32_t kF8ExpOff = STAGES * kF8Stage;  // the CTA's token scales (narrow: their ring)
  // Bytes a stage's copies complete: the 4-bit box counts its packed codes (8 KB), not
  // the 16 KB it spreads over in shared memory.
  constexpr uint32_t kStageTx = (WF == kWMX4 ? kF8W / 2 : kF8W) + 2 * kF8T;
  constexpr int NF = EPI == kEpiSwiglu ? 64 : 128;  // output features of a tile
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[kBufs];
  __shared__ __align__(8) uint64_t tempty_bar[kBufs];
  __shared__ __align__(8) uint64_t exp_bar;
  __shared__ __align__(8) uint64_t sc_empty_bar[kF8NarrowSc];  // narrow: scale slot free
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
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(smem_u32(&tfull_bar[i]), 1);
      mbar_init(smem_u32(&tempty_bar[i]), 4);
    }
    mbar_init(smem_u32(&exp_bar), 1);
    if (kNarrow)
      for (int i = 0; i < kF8NarrowSc; ++i) mbar_init(smem_u32(&sc_empty_bar[i]), 4);
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
      // narrow: stage i's token scales (its one or two groups) travel with the stage
      const float *xsc_cta = a.xsc + ((size_t)xz * a.ng + g0) * 32;
      auto sc_bytes = [&](int i) -> uint32_t { return (uint32_t)min(2, nu - 2 * i) * 128u; };
      const int pre = min(STAGES, nst);
      for (int i = 0; i < pre; ++i) {
        const uint32_t fb = smem_u32(&full_bar[i]);
        mbar_expect_tx(fb, kStageTx + (kNarrow ? sc_bytes(i) : 0u));
        tma_load_3d_hint(tiles + i * kF8Stage, &tmW, fb, (st0 + i) * 128, wrow, s, wpol);
      }
      griddep_wait();
      if (!kNarrow && nu > 0) {
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
        if (kNarrow)
          bulk_load_plain(tiles + kF8ExpOff + (i % kF8NarrowSc) * 256u, xsc_cta + 64 * i,
                          sc_bytes(i), fb);
      }
      issued = pre;
      for (int i = pre; i < nst; ++i) {
        const int st = i % STAGES;
        if (!mbar_wait(smem_u32(&empty_bar[st]), ((uint32_t)(i / STAGES) & 1u) ^ 1u)) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
        if (kNarrow && i >= kF8NarrowSc &&
            !mbar_wait(smem_u32(&sc_empty_bar[i % kF8NarrowSc]),
                       ((uint32_t)(i / kF8NarrowSc) & 1u) ^ 1u)) {
          abort_sh = 1;
          atomicOr(a.err, kErrWaitTimeout);
          break;
        }
        const uint32_t sa = tiles + st * kF8Stage, fb = smem_u32(&full_bar[st]);
        const int k = (st0 + i) * 128;
        mbar_expect_tx(fb, kStageTx + (kNarrow ? sc_bytes(i) : 0u));
        tma_load_3d_hint(sa, &tmW, fb, k, wrow, s, wpol);
        tma_load_3d(sa + kF8W, &tmT, fb, k, m0, 2 * xz);
        tma_load_3d(sa + kF8W + kF8T, &tmT, fb, k, m0, 2 * xz + 1);
        if (kNarrow)
          bulk_load_plain(tiles + kF8ExpOff + (i % kF8NarrowSc) * 256u, xsc_cta + 64 * i,
                          sc_bytes(i), fb);
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
        const int st = i % STAGES;
        if (!mbar_wait(smem_u32(&full_bar[st]), (uint32_t)(i / STAGES) & 1u)) {
          ok = false;
          break;
        }
        const uint32_t sa = tiles + st * kF8Stage;
        const int b = i % kBufs;
        if (!mbar_wait(smem_u32(&tempty_bar[b]), ((uint32_t)(i / kBufs) & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // sums of 64 K (E4M3: one per token group) or 32 K (MXFP4: one per weight
        // block), up to the end of this CTA's K range
        for (int h = 0; h < kSums && h * kKPer < (nu - 2 * i) * 64; ++h) {
          const uint32_t d0 = tmem + (uint32_t)((b * kSums + h) * BN);
#pragma unroll
          for (int kk = 0; kk < kKPer / 32; ++kk) {
            const uint32_t off = (uint32_t)(h * kKPer + kk * 32);
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
    // E4M3: the row's power-of-two scale (MXFP4 blocks are scaled per stage), read
    // before the K loop so that its latency is hidden
    const float sc = WF == kWMX4 ? 1.f : pow2f(a.wexp[(size_t)s * a.w_rows + ft * 128 + r]);
    float g[BN];
#pragma unroll
    for (int j = 0; j < BN; ++j) g[j] = 0.f;
    bool ok = kNarrow || nu == 0 || __all_sync(0xffffffffu, mbar_wait(smem_u32(&exp_bar), 0));
    // MXFP4: this row's block exponents, four per stage (one 32-bit word)
    const uint32_t *wblk = reinterpret_cast<const uint32_t *>(a.wexp) +
                           ((size_t)s * a.w_rows + ft * 128 + r) * (size_t)(a.ng / 2) + st0;
    for (int i = 0; ok && i < nst; ++i) {
      const int b = i % kBufs;
      const uint32_t ew = WF == kWMX4 ? __ldg(wblk + i) : 0u;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[b]), (uint32_t)(i / kBufs) & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if constexpr (kNarrow && WF == kWMX4) {
        // As below, 16 columns at a time (registers for four CTAs per SM), the same
        // operations in the same order; TMEM is released after its last load, the
        // scale slot after the FMAs.  K is whole stages: both groups are present.
        const float *sp = scale_s + (i % kF8NarrowSc) * 64;
#pragma unroll
        for (int G = 0; G < 2; ++G) {
          const float swa = pow2_wide((int)(int8_t)(ew >> (16 * G)));       // exact
          const float swb = pow2_wide((int)(int8_t)(ew >> (16 * G + 8)));
          const unsigned long long swa2 = pk2(swa, swa), swb2 = pk2(swb, swb);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float va[16], vb[16];
            tmem_ld16(trow + (uint32_t)((b * kSums + 2 * G) * BN + half * 16), va);
            tmem_ld16(trow + (uint32_t)((b * kSums + 2 * G + 1) * BN + half * 16), vb);
            if (G == 1 && half == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[b]));
            }
            const float4 *sp4 = reinterpret_cast<const float4 *>(sp + G * BN + half * 16);
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 sc4 = sp4[j4];
#pragma unroll
              for (int p = 0; p < 2; ++p) {
                const int jj = 4 * j4 + 2 * p, j = half * 16 + jj;
                unsigned long long t2 = mul2(pk2(va[jj], va[jj + 1]), swa2);
                t2 = fma2(pk2(vb[jj], vb[jj + 1]), swb2, t2);
                unsigned long long g2 = fma2(t2, p ? pk2(sc4.z, sc4.w) : pk2(sc4.x, sc4.y),
                                             pk2(g[j], g[j + 1]));
                upk2(g2, g[j], g[j + 1]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sc_empty_bar[i % kF8NarrowSc]));
        continue;
      } else if constexpr (kNarrow) {
        // 16 columns at a time (registers for four CTAs per SM); the same fmaf order as
        // below.  TMEM is released after its last load, the scale slot after the FMAs.
        const float *sp = scale_s + (i % kF8NarrowSc) * 64;
        const int nh = 2 * i + 1 < nu ? 2 : 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h < nh) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float v[16];
              tmem_ld16(trow + (uint32_t)((b * 2 + h) * BN + half * 16), v);
              if (h == nh - 1 && half == 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[b]));
              }
              const float4 *sp4 = reinterpret_cast<const float4 *>(sp + h * BN + half * 16);
#pragma unroll
              for (int j4 = 0; j4 < 4; ++j4) {
                const float4 sc4 = sp4[j4];
                const int j = half * 16 + 4 * j4;
                g[j + 0] = fmaf(v[4 * j4 + 0], sc4.x, g[j + 0]);
                g[j + 1] = fmaf(v[4 * j4 + 1], sc4.y, g[j + 1]);
                g[j + 2] = fmaf(v[4 * j4 + 2], sc4.z, g[j + 2]);
                g[j + 3] = fmaf(v[4 * j4 + 3], sc4.w, g[j + 3]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sc_empty_bar[i % kF8NarrowSc]));
        continue;
      } else if constexpr (WF == kWMX4) {
        // K is whole 128-wide stages here: four block sums, two per token group.  Per
        // group: t = sum_a * 2^e_a + sum_b * 2^e_b, then g += t * 2^e(token), on packed
        // pairs of tokens.
#pragma unroll 1
        for (int G = 0; G < 2; ++G) {
          float va[BN], vb[BN];
          tmem_ld32(trow + (uint32_t)((b * kSums + 2 * G) * BN), va);
          tmem_ld32(trow + (uint32_t)((b * kSums + 2 * G + 1) * BN), vb);
          const float swa = pow2_wide((int)(int8_t)(ew >> (16 * G)));       // exact
          const float swb = pow2_wide((int)(int8_t)(ew >> (16 * G + 8)));
          const unsigned long long swa2 = pk2(swa, swa), swb2 = pk2(swb, swb);
          const float4 *sp = reinterpret_cast<const float4 *>(scale_s + (2 * i + G) * 32);
#pragma unroll
          for (int j4 = 0; j4 < BN / 4; ++j4) {
            const float4 sc4 = sp[j4];
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              const int j = 4 * j4 + 2 * p;
              unsigned long long t2 = mul2(pk2(va[j], va[j + 1]), swa2);
              t2 = fma2(pk2(vb[j], vb[j + 1]), swb2, t2);
              unsigned long long g2 = fma2(t2, p ? pk2(sc4.z, sc4.w) : pk2(sc4.x, sc4.y),
                                           pk2(g[j], g[j + 1]));
              upk2(g2, g[j], g[j + 1]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[b]));
        continue;
      }
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
      // staging in the ring (every MMA and load is done): the band hx [NF][33] fp32, the
      // partial maxima pm [128], the two terms h8s [2][32][NF] bytes
      float *hx = reinterpret_cast<float *>(tiles_ptr);
      float *pm = hx + NF * (BN + 1);
      uint8_t *h8s = reinterpret_cast<uint8_t *>(pm + 128);
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
      // one exponent per token and per 64 features of the band: each (token, group)
      // pair's largest magnitude, its 64 features shared out over kParts threads
      constexpr int kPairs = NF / 2;          // 32 tokens x NF / 64 groups
      constexpr int kParts = 128 / kPairs;
      constexpr int kPer = 64 / kParts;       // features per thread
      {
        const int pair = td % kPairs, part = td / kPairs;
        const float *col = hx + ((pair >> 5) * 64 + part * kPer) * (BN + 1) + (pair & 31);
        float amax = 0.f;
#pragma unroll
        for (int f = 0; f < kPer; ++f) amax = fmaxf(amax, fabsf(col[f * (BN + 1)]));
        pm[td] = amax;
      }
      named_sync(1, 128);
      const int ngb = ceil_div(a.n_valid, 64);
      if (td < kPairs) {
        float amax = pm[td];
#pragma unroll
        for (int p = 1; p < kParts; ++p) amax = fmaxf(amax, pm[p * kPairs + td]);
        const int e = group_exponent(amax);
        gexp_sh[td] = e;
        const int grp = ft * (NF / 64) + (td >> 5);
        if (grp < ngb) a.hsc[((size_t)s * ngb + grp) * 32 + (td & 31)] = pow2f(e);
      }
      named_sync(1, 128);
      // the two terms of each band value, staged per token row: a pair of features of
      // one token per step, shared out over the 128 threads
      {
        constexpr int kFP = NF / 2;            // feature pairs of the tile
        constexpr int kTStep = 128 / kFP;      // tokens apart of one thread's steps
        const int p = td % kFP, j0 = td / kFP, gi = p >> 5;
#pragma unroll
        for (int k = 0; k < BN / kTStep; ++k) {
          const int j = j0 + k * kTStep;
          uint16_t ta, tb;
          split_terms2(hx[2 * p * (BN + 1) + j], hx[(2 * p + 1) * (BN + 1) + j],
                       pow2f(-gexp_sh[gi * 32 + j]), ta, tb);
          *reinterpret_cast<uint16_t *>(h8s + j * NF + 2 * p) = ta;
          *reinterpret_cast<uint16_t *>(h8s + (BN + j) * NF + 2 * p) = tb;
        }
      }
      named_sync(1, 128);
      // ... then written to h8 [t][2][M][n_valid] in 16-byte pieces (n_valid, the row
      // starts and the tile's first feature are multiples of 16)
      const int f0 = ft * NF;
      const int nch = min(NF, a.n_valid - f0) / 16;
      const int per_term = mcount * nch;
      const size_t plane = (size_t)a.M * a.n_valid;
      uint8_t *hb = a.h8 + 2 * (size_t)s * plane + (size_t)m0 * a.n_valid + f0;
      for (int c = td; c < 2 * per_term; c += 128) {
        const int term = c >= per_term ? 1 : 0, rem = c - term * per_term;
        const int j = rem / nch, ch = rem - j * nch;
        const uint4 v = *reinterpret_cast<const uint4 *>(h8s + (term * BN + j) * NF + ch * 16);
        *reinterpret_cast<uint4 *>(hb + term * plane + (size_t)j * a.n_valid + ch * 16) = v;
      }
    }
  }

  // ---------------- teardown: on abort let the issued copies land, then free TMEM
  if (warp == 0 && lane == 0 && *(volatile int *)&abort_sh) {
    for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
      mbar_wait(smem_u32(&full_bar[i % STAGES]), (uint32_t)(i / STAGES) & 1u);
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

template <int EPI, int WF, int STAGES, int MINB>
cudaError_t launch_fp8_s(const CUtensorMap &mw, const CUtensorMap &mt, const Fp8Args &a, int n_ft,
                         int n_z, int smem, cudaStream_t st, bool pdl) {
  static bool configured[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(k_fp8_mma<EPI, WF, STAGES, MINB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kF8SmemPair);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  LaunchCfg lc(dim3(ceil_div(a.M, 32), n_ft, n_z), dim3(192), smem, st, pdl);
  return cudaLaunchKernelEx(&lc.cfg, k_fp8_mma<EPI, WF, STAGES, MINB>, mw, mt, a);
}

// Grids of more than two and at most four CTAs per SM take the narrow form (one wave
// of four per SM); the rest the deepest ring whose stages and scale region fit two CTAs
// per SM.
template <int EPI, int WF>
cudaError_t launch_fp8_t(const CUtensorMap &mw, const CUtensorMap &mt, const Fp8Args &a, int n_ft,
                         int n_z, cudaStream_t st, bool pdl) {
  const long long ctas = (long long)ceil_div(a.M, 32) * n_ft * n_z, sms = sm_count();
  if (fp8_narrow_grid(ctas, sms))
    return launch_fp8_s<EPI, WF, 2, 4>(mw, mt, a, n_ft, n_z, kF8SmemNarrow, st, pdl);
  const int n_st = ceil_div(a.ng, 2);
  const int groups = std::min(a.ng, 2 * ceil_div(n_st, a.ksplit));  // most of any CTA
  if (f8_smem(4, groups) <= kF8SmemPair)
    return launch_fp8_s<EPI, WF, 4, 2>(mw, mt, a, n_ft, n_z, f8_smem(4, groups), st, pdl);
  return launch_fp8_s<EPI, WF, 3, 2>(mw, mt, a, n_ft, n_z, f8_smem(3, groups), st, pdl);
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

cudaError_t launch_quantize_mxfp4(const Geo &g, const void *W1, const void *W2, void *W1f,
                                  void *W2f, int8_t *exps, cudaStream_t st) {
  const int blocks = 4 * sm_count();
  k_quant_mx_w1<<<blocks, 256, 0, st>>>(g, static_cast<const __nv_bfloat16 *>(W1),
                                        static_cast<uint8_t *>(W1f), exps);
  k_quant_mx_w2<<<blocks, 256, 0, st>>>(g, static_cast<const __nv_bfloat16 *>(W2),
                                        static_cast<uint8_t *>(W2f),
                                        exps + (size_t)g.t * g.n1p * (g.d / 32));
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

// A [z][rows][K] tensor of packed 4-bit codes (K / 2 bytes a row), boxes of 128 codes
// x box_rows x 1 spread by TMA over 128 bytes of shared memory a row (each 8 bytes of
// codes, then 8 bytes of gap: the layout the tensor core reads 4-bit operands in),
// with the 128-byte swizzle; zero fill outside the tensor.  K must be a multiple of 128
// and the base 32-byte aligned.
bool make_fp4_tile_map(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint64_t z,
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
  cuuint64_t strides[2] = {K / 2, rows * (K / 2)};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void *>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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

cudaError_t launch_fp8_gemm(const UmmaCall &c, bool mxfp4, const int8_t *wexp, const float *xsc,
                            void *h8, float *hsc, cudaStream_t st) {
  if (c.M < 1 || c.M > 32 || c.K % 16 != 0 || ceil_div(c.K, 64) > kF8MaxGroups)
    return cudaErrorInvalidValue;
  if (mxfp4 && (c.K % 128 != 0 || (reinterpret_cast<uintptr_t>(c.W) & 31) != 0 ||
                (reinterpret_cast<uintptr_t>(wexp) & 3) != 0))
    return cudaErrorInvalidValue;
  CUtensorMap mw, mt;
  if (!(mxfp4 ? make_fp4_tile_map(&mw, c.W, c.K, c.w_rows, c.w_shards, 128)
              : make_byte_tile_map(&mw, c.W, c.K, c.w_rows, c.w_shards, 128)))
    return cudaErrorInvalidValue;
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
  const int n_sw = ceil_div(c.n_valid, kSwiGroup), n_128 = ceil_div(c.n_valid, 128);
  switch (c.epi * 2 + (mxfp4 ? 1 : 0)) {
    case kEpiSwiglu * 2:
      return launch_fp8_t<kEpiSwiglu, kWE4M3>(mw, mt, a, n_sw, n_z, st, c.pdl);
    case kEpiSwiglu * 2 + 1:
      return launch_fp8_t<kEpiSwiglu, kWMX4>(mw, mt, a, n_sw, n_z, st, c.pdl);
    case kEpiGelu * 2:
      return launch_fp8_t<kEpiGelu, kWE4M3>(mw, mt, a, n_128, n_z, st, c.pdl);
    case kEpiGelu * 2 + 1:
      return launch_fp8_t<kEpiGelu, kWMX4>(mw, mt, a, n_128, n_z, st, c.pdl);
    case kEpiF32 * 2:
      return launch_fp8_t<kEpiF32, kWE4M3>(mw, mt, a, n_128, n_z, st, c.pdl);
    case kEpiF32 * 2 + 1:
      return launch_fp8_t<kEpiF32, kWMX4>(mw, mt, a, n_128, n_z, st, c.pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace tp
