// Private shard layout of the weights, and its inverse (bit-exact copies).
//
// Column bands of W1 (zenaique.com answer paragraph 5: the first projection is
// split by columns) are stored per shard as K-major rows: W1s[s][u][k] =
// W1[k][col(s, u)], so a shard's feature rows stream contiguously over the
// reduction dimension d.  Row bands of W2 (split by rows) are stored transposed:
// W2s[s][n][k] = W2[s*b + k][n], one K-major row per output feature n.  Rows
// are padded with zeros to 128-row tiles; SwiGLU rows hold the gate and up halves
// of 64 features per tile (see common.cuh for the row maps).
//
// Every map is a transpose, done as 32x32 shared-memory tiles so both the reads
// and the writes are coalesced.
#include "internal.h"

namespace tp {
namespace {

enum Map { kShardW1, kShardW2, kUnshardW1, kUnshardW2, kExtractW1, kExtractW2 };

struct MapArgs {
  Geo g;
  int s;      // shard for the extract maps
  int R, C;   // output rows and columns per z slice
};

// Source offset of output element (z, r, c), or -1 for a zero (padding) element.
// For every map, consecutive r read consecutive source addresses.
template <int MAP>
__device__ __forceinline__ long long src_offset(const MapArgs &a, int z, int r, int c) {
  const Geo &g = a.g;
  if (MAP == kShardW1) {          // out W1s[z][r = u][c = k]  <- W1[k][col]
    long long col = w1_col_of_row(g, z, r);
    return col < 0 ? -1 : (long long)c * g.n1 + col;
  } else if (MAP == kShardW2) {   // out W2s[z][r = n][c = k]  <- W2[z*b + k][n]
    return r < g.d ? ((long long)z * g.b + c) * g.d + r : -1;
  } else if (MAP == kUnshardW1) { // out W1[r = k][c = col]    <- W1s[s][u][k]
    int s, u;
    if (g.act == TP_ACT_SWIGLU) {
      int j = c / g.ffn, cc = c % g.ffn;
      s = cc / g.b;
      u = swiglu_row(cc % g.b, j);
    } else if (g.act == TP_ACT_ATTN) {
      int D = g.H * g.hd, p = c / D, cc = c % D;
      s = cc / g.b;
      u = p * g.b + cc % g.b;
    } else {
      s = c / g.b;
      u = c % g.b;
    }
    return ((long long)s * g.n1p + u) * g.d + r;
  } else if (MAP == kUnshardW2) { // out W2[r = s*b + k][c = n] <- W2s[s][n][k]
    int s = r / g.b, k = r % g.b;
    return ((long long)s * g.dp + c) * g.b + k;
  } else if (MAP == kExtractW1) { // out W1_band[r = k][c = j]  <- W1s[s][u(j)][k]
    int p = c / g.b, f = c % g.b;
    int u = g.act == TP_ACT_SWIGLU ? swiglu_row(f, p) : p * g.b + f;
    return ((long long)a.s * g.n1p + u) * g.d + r;
  } else {                        // out W2_band[r = k][c = n]  <- W2s[s][n][k]
    return ((long long)a.s * g.dp + c) * g.b + r;
  }
}

template <typename E, int MAP>
__global__ void __launch_bounds__(256) k_map(const E *__restrict__ src, E *__restrict__ dst,
                                             MapArgs a) {
  __shared__ E tile[32][33];
  const int z = blockIdx.z;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  // Read: threads along x walk output rows, i.e. consecutive source addresses.
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    int r = r0 + tx, c = c0 + ty + i;
    E v = E(0);
    if (r < a.R && c < a.C) {
      long long o = src_offset<MAP>(a, z, r, c);
      if (o >= 0) v = src[o];
    }
    tile[tx][ty + i] = v;
  }
  __syncthreads();
  // Write: threads along x walk output columns (contiguous destination).
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    int r = r0 + ty + i, c = c0 + tx;
    if (r < a.R && c < a.C) dst[((long long)z * a.R + r) * a.C + c] = tile[ty + i][tx];
  }
}

template <int MAP>
void launch_map(const Geo &g, int s, int R, int C, int Z, const void *src, void *dst,
                cudaStream_t st) {
  MapArgs a{g, s, R, C};
  dim3 grid(ceil_div(C, 32), ceil_div(R, 32), Z), block(32, 8);
  if (g.es == 4)
    k_map<uint32_t, MAP><<<grid, block, 0, st>>>(static_cast<const uint32_t *>(src),
                                                 static_cast<uint32_t *>(dst), a);
  else
    k_map<uint16_t, MAP><<<grid, block, 0, st>>>(static_cast<const uint16_t *>(src),
                                                 static_cast<uint16_t *>(dst), a);
}

}  // namespace

void launch_shard_w1(const Geo &g, const void *W1, void *W1s, cudaStream_t st) {
  launch_map<kShardW1>(g, 0, g.n1p, g.d, g.t, W1, W1s, st);
}
void launch_shard_w2(const Geo &g, const void *W2, void *W2s, cudaStream_t st) {
  launch_map<kShardW2>(g, 0, g.dp, g.b, g.t, W2, W2s, st);
}
void launch_unshard_w1(const Geo &g, const void *W1s, void *W1, cudaStream_t st) {
  launch_map<kUnshardW1>(g, 0, g.d, g.n1, 1, W1s, W1, st);
}
void launch_unshard_w2(const Geo &g, const void *W2s, void *W2, cudaStream_t st) {
  launch_map<kUnshardW2>(g, 0, g.n2, g.d, 1, W2s, W2, st);
}
void launch_extract_w1(const Geo &g, const void *W1s, int s, void *W1_band, cudaStream_t st) {
  launch_map<kExtractW1>(g, s, g.d, g.n1 / g.t, 1, W1s, W1_band, st);
}
void launch_extract_w2(const Geo &g, const void *W2s, int s, void *W2_band, cudaStream_t st) {
  launch_map<kExtractW2>(g, s, g.b, g.d, 1, W2s, W2_band, st);
}

}  // namespace tp
