// Block-level helpers shared by the kernels that finish the routing (1024 threads):
// a column-wise scan of per-block expert counts, and the expert layout of the
// permuted buffers (offsets and each expert's first GEMM row tile) from per-expert
// row counts.
#pragma once

#include <stdint.h>

#include "internal.h"

namespace moe {

// blk[nblk][N] holds per-block counts of every expert. Replaces each count by the
// number of the same expert's entries in earlier blocks (exclusive bases) and writes
// the column totals to s_total[N]. Thread (g, col) walks a contiguous range of rows
// of one column; a warp covers consecutive columns of the same rows, so its loads
// are coalesced, and a prefix over the row groups gives every group its base (a fixed
// pattern, so the result does not depend on scheduling). Contains __syncthreads.
__device__ inline void column_scan(int32_t* blk, int nblk, int N, int32_t* s_total) {
  __shared__ int32_t ip[1024];
  const int tid = threadIdx.x;
  int np2 = 1;
  while (np2 < N) np2 <<= 1;
  const int G = 1024 / np2;
  const int col = tid % np2, g = tid / np2;
  const int R = (nblk + G - 1) / G;
  const int r0 = min(nblk, g * R), r1 = min(nblk, r0 + R);
  // The first RC rows stay in registers for the second pass; more rows are reloaded.
  constexpr int RC = 16, B = 8;
  int cache[RC];
  int isum = 0;
  if (col < N) {
#pragma unroll
    for (int u = 0; u < RC; ++u) cache[u] = r0 + u < r1 ? blk[(size_t)(r0 + u) * N + col] : 0;
#pragma unroll
    for (int u = 0; u < RC; ++u) isum += cache[u];
    for (int rb = r0 + RC; rb < r1; rb += B) {
      int iv[B];
#pragma unroll
      for (int u = 0; u < B; ++u) iv[u] = rb + u < r1 ? blk[(size_t)(rb + u) * N + col] : 0;
#pragma unroll
      for (int u = 0; u < B; ++u) isum += iv[u];
    }
  }
  ip[tid] = isum;
  __syncthreads();
  for (int d = 1; d < G; d <<= 1) {
    const int iv = g >= d ? ip[tid - d * np2] : 0;
    __syncthreads();
    ip[tid] += iv;
    __syncthreads();
  }
  if (col < N && g == G - 1) s_total[col] = ip[tid];
  if (col < N) {
    int run = ip[tid] - isum;
#pragma unroll
    for (int u = 0; u < RC; ++u) {
      if (r0 + u < r1) blk[(size_t)(r0 + u) * N + col] = run;
      run += cache[u];
    }
    for (int rb = r0 + RC; rb < r1; rb += B) {
      int iv[B];
#pragma unroll
      for (int u = 0; u < B; ++u) iv[u] = rb + u < r1 ? blk[(size_t)(rb + u) * N + col] : 0;
#pragma unroll
      for (int u = 0; u < B; ++u) {
        if (rb + u < r1) blk[(size_t)(rb + u) * N + col] = run;
        run += iv[u];
      }
    }
  }
  __syncthreads();
}

// Where every expert's rows go: offsets[e] = rows of the experts before e, and for
// 128-row [0] and 256-row [1] tiles the first tile of each expert and the tile count
// (the expert GEMMs find a tile's expert and first row from these). s_rows[Ntot]: rows
// per expert (shared memory). Warp 0 does the work; every thread may call it.
struct ExpertLayout {
  int32_t* offsets;          // [Ntot+1]
  int32_t* tile_first[2];    // [Ntot+1]
  int32_t* num_mtiles[2];    // [1]
};

__device__ inline void layout_experts(const int32_t* s_rows, int Ntot, const ExpertLayout& o) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int per = (Ntot + 31) / 32;  // experts per lane, <= 9
  const int e0 = min(Ntot, lane * per), e1 = min(Ntot, e0 + per);
  int off = 0, t1 = 0, t2 = 0;
  for (int e = e0; e < e1; ++e) {
    off += s_rows[e];
    t1 += (s_rows[e] + TILE_ROWS_1 - 1) / TILE_ROWS_1;
    t2 += (s_rows[e] + TILE_ROWS_2 - 1) / TILE_ROWS_2;
  }
  int xo = off, x1 = t1, x2 = t2;  // inclusive scans over the lanes
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int po = __shfl_up_sync(0xffffffffu, xo, d);
    const int p1 = __shfl_up_sync(0xffffffffu, x1, d);
    const int p2 = __shfl_up_sync(0xffffffffu, x2, d);
    if (lane >= d) {
      xo += po;
      x1 += p1;
      x2 += p2;
    }
  }
  int ofs = xo - off, a1 = x1 - t1, a2 = x2 - t2;
  for (int e = e0; e < e1; ++e) {
    o.tile_first[0][e] = a1;
    o.tile_first[1][e] = a2;
    o.offsets[e] = ofs;
    ofs += s_rows[e];
    a1 += (s_rows[e] + TILE_ROWS_1 - 1) / TILE_ROWS_1;
    a2 += (s_rows[e] + TILE_ROWS_2 - 1) / TILE_ROWS_2;
  }
  if (lane == 31) {
    o.offsets[Ntot] = xo;
    o.tile_first[0][Ntot] = x1;
    o.tile_first[1][Ntot] = x2;
    *o.num_mtiles[0] = x1;
    *o.num_mtiles[1] = x2;
  }
}

}  // namespace moe
