// The routing decisions' block-level reductions and the work of the block that
// finishes last (the per-expert scan over the blocks, capacity, losses and the expert
// layout), shared by the routing-decision kernels. The formulas and their sources are
// stated where the kernels are (route_select.cu).
#pragma once

#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "expert_layout.cuh"
#include "internal.h"

namespace moe {
namespace route {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Exclusive prefix of v over the threads of the block (a multiple of 32), in thread
// order; *total gets the sum. s_w: 32 ints of shared memory. Contains __syncthreads.
__device__ inline int block_exclusive_scan(int v, int32_t* s_w, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? s_w[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    if (lane < nw) s_w[lane] = w;
  }
  __syncthreads();
  const int before = (warp > 0 ? s_w[warp - 1] : 0) + x - v;
  *total = s_w[nw - 1];
  __syncthreads();
  return before;
}

// Sum of v over the block in a fixed order (deterministic). s_d: 32 doubles.
__device__ inline double block_sum(double v, double* s_d) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  v = warp_sum(v);
  if (lane == 0) s_d[warp] = v;
  __syncthreads();
  double r = warp_sum(lane < nw ? s_d[lane] : 0.0);
  __syncthreads();
  return r;
}

// The last block's work (any block of NT >= 256 threads, NT a power of two times 32 up
// to 1024). Thread (g, col) walks a contiguous range of block rows of one expert
// column; a warp covers consecutive columns of the same rows, so its loads are
// coalesced. A parallel prefix over the row groups gives every group its base, and
// warp 0 scans the experts for offsets and tile starts.
__device__ inline void finish_routing(const SelectArgs& a, int nblk) {
  __shared__ int32_t ip[1024];
  __shared__ float fq[1024];
  __shared__ int32_t s_counts[MAX_EXPERTS], s_kept[MAX_EXPERTS];
  __shared__ float s_psum[256];
  __shared__ int32_t s_w[32];
  __shared__ double s_d[32];
  const int tid = threadIdx.x;
  const int NT = blockDim.x;
  const int N = a.N, Ntot = a.N + a.S;
  // Valid tokens: per-block counts -> exclusive bases, and their total.
  int T_valid = a.T;
  if (a.valid != nullptr) {
    const int R = (nblk + NT - 1) / NT;
    const int b0 = min(nblk, tid * R), b1 = min(nblk, b0 + R);
    int mine = 0;
    for (int b = b0; b < b1; ++b) mine += a.blk_valid[b];
    int run = block_exclusive_scan(mine, s_w, &T_valid);
    for (int b = b0; b < b1; ++b) {
      const int c = a.blk_valid[b];
      a.blk_valid[b] = run;
      run += c;
    }
  }
  // Capacity of this call: C = ceil(CF * T_valid * k / N) in double, at most T_valid*k
  // (the host's value when every token is valid). One thread evaluates it (fp64 is
  // slow on this part) and shares it; the first read comes after the barrier that
  // follows the column sums below.
  __shared__ long long s_C;
  if (tid == 0) {
    long long C = a.C;
    if (a.valid != nullptr && a.cf > 0.0) {
      const double c = ceil(a.cf * (double)T_valid * (double)a.k / (double)N);
      const double slots = (double)T_valid * (double)a.k;
      C = c >= slots ? (long long)slots : (long long)c;
    }
    s_C = C;
    *a.cap = (int32_t)C;
  }
  double d2 = 0.0;  // sum of (P - 1/N)^2 over the valid tokens
  if (a.aux_std2 != nullptr) {
    const int R = (nblk + NT - 1) / NT;
    const int b0 = min(nblk, tid * R), b1 = min(nblk, b0 + R);
    double mine = 0.0;
    for (int b = b0; b < b1; ++b) mine += (double)a.blk_d2[b];
    d2 = block_sum(mine, s_d);
  }
  int np2 = 1;
  while (np2 < N) np2 <<= 1;
  const int G = NT / np2;                   // row groups (NT >= N)
  const int col = tid % np2, g = tid / np2;
  const int R = (nblk + G - 1) / G;
  const int r0 = min(nblk, g * R), r1 = min(nblk, r0 + R);
  // The first RC rows of counts stay in registers for the second pass; more rows are
  // loaded in batches of B (B loads in flight per thread) and reloaded.
  constexpr int RC = 8, B = 8;
  int cache[RC];
  int isum = 0;
  float fsum = 0.f;
  if (col < N) {
    float fc[RC];
#pragma unroll
    for (int u = 0; u < RC; ++u) {
      const bool in = r0 + u < r1;
      cache[u] = in ? a.blk_counts[(size_t)(r0 + u) * N + col] : 0;
      fc[u] = in ? a.blk_psum[(size_t)(r0 + u) * N + col] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < RC; ++u) {
      isum += cache[u];
      fsum += fc[u];
    }
    for (int rb = r0 + RC; rb < r1; rb += B) {
      int iv[B];
      float fv[B];
#pragma unroll
      for (int u = 0; u < B; ++u) {
        const bool in = rb + u < r1;
        iv[u] = in ? a.blk_counts[(size_t)(rb + u) * N + col] : 0;
        fv[u] = in ? a.blk_psum[(size_t)(rb + u) * N + col] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < B; ++u) {
        isum += iv[u];
        fsum += fv[u];
      }
    }
  }
  ip[tid] = isum;
  fq[tid] = fsum;
  __syncthreads();
  // inclusive prefix over the row groups of each column (fixed pattern: deterministic)
  for (int d = 1; d < G; d <<= 1) {
    const int iv = g >= d ? ip[tid - d * np2] : 0;
    const float fv = g >= d ? fq[tid - d * np2] : 0.f;
    __syncthreads();
    ip[tid] += iv;
    fq[tid] += fv;
    __syncthreads();
  }
  const long long C = s_C;
  if (col < N && g == G - 1) {
    const int run = ip[tid];
    const int kept = (C < 0 || (long long)run <= C) ? run : (int)C;
    s_counts[col] = run;
    s_kept[col] = kept;
    s_psum[col] = fq[tid];
    a.counts[col] = run;
    a.kept[col] = kept;
    if (a.user_counts != nullptr) a.user_counts[col] = run;
    if (a.user_kept != nullptr) a.user_kept[col] = kept;
  }
  if (tid < a.S) {  // shared experts take every valid token, no capacity
    s_counts[N + tid] = T_valid;
    s_kept[N + tid] = T_valid;
    a.counts[N + tid] = T_valid;
    a.kept[N + tid] = T_valid;
  }
  if (col < N) {  // exclusive per-expert base of every block
    int run = ip[tid] - isum;
#pragma unroll
    for (int u = 0; u < RC; ++u) {
      if (r0 + u < r1) a.blk_counts[(size_t)(r0 + u) * N + col] = run;
      run += cache[u];
    }
    for (int rb = r0 + RC; rb < r1; rb += B) {
      int iv[B];
#pragma unroll
      for (int u = 0; u < B; ++u)
        iv[u] = rb + u < r1 ? a.blk_counts[(size_t)(rb + u) * N + col] : 0;
#pragma unroll
      for (int u = 0; u < B; ++u) {
        if (rb + u < r1) a.blk_counts[(size_t)(rb + u) * N + col] = run;
        run += iv[u];
      }
    }
  }
  __syncthreads();
  if (tid < 32) {  // warp 0: the losses over the routed experts
    const int lane = tid;
    float fp = 0.f;
    double lsum = 0.0;
    int empty = 0;
    for (int e = lane; e < N; e += 32) {
      fp = fmaf((float)s_counts[e], s_psum[e], fp);
      if (a.aux_kl != nullptr) {
        if (s_counts[e] == 0) empty = 1;
        else lsum += log((double)N * (double)s_counts[e] / ((double)T_valid * (double)a.k));
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) fp += __shfl_xor_sync(0xffffffffu, fp, d);
    if (a.aux_kl != nullptr) {
      lsum = warp_sum(lsum);
      empty = __any_sync(0xffffffffu, empty);
    }
    if (lane == 0) {
      // aux = N * sum_e (counts_e / (T*k)) * (Psum_e / T), T the valid tokens;
      // counts <= T*k and sum_e Psum_e = T keep every term well inside fp32 range
      const float Tf = (float)T_valid;
      *a.aux = T_valid > 0 ? (float)N * (fp / (Tf * (float)a.k)) / Tf : 0.f;
      // KL(uniform || f) = -(1/N) sum_e log(N f_e); +inf when an expert got nothing
      if (a.aux_kl != nullptr)
        *a.aux_kl = T_valid == 0 ? 0.f : empty ? INFINITY : (float)(-lsum / (double)N);
      // unbiased variance of the T_valid*N probabilities around their mean 1/N
      if (a.aux_std2 != nullptr)
        *a.aux_std2 =
            T_valid == 0 ? 0.f : (float)(d2 / ((double)T_valid * (double)N - 1.0));
    }
  }
  ExpertLayout lay;
  lay.offsets = a.offsets;
  for (int tb = 0; tb < 2; ++tb) {
    lay.tile_first[tb] = a.tile_first[tb];
    lay.num_mtiles[tb] = a.num_mtiles[tb];
  }
  layout_experts(s_kept, Ntot, lay);
}

// The same finish for small layers in one warp, with no block barrier, where
// warp_finish_fits() holds (internal.h). Up to 32 experts, L = 32 / np2(N) lanes share
// an expert column, each taking a contiguous range of block rows, and a prefix over
// those ranges (shuffles) gives every block its base. Above 32 experts a lane takes
// all rows of experts lane, lane + 32, ... one after another. Lane e then holds expert
// e's totals (e, e + 32, ... above 32 experts), so the aux sum reduces the same
// per-expert products in the same order as the block finish. The kernels take the
// finish as a template argument chosen on the host, so each carries the code of one
// finish only.
// Called by warp 0 only; MAXR is the max_rows that warp_finish_fits() was given.
template <int MAXR>
__device__ inline void finish_routing_warp(const SelectArgs& a, int nblk) {
  __shared__ int32_t s_rows[MAX_EXPERTS];
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x;
  const int N = a.N, Ntot = a.N + a.S;
  int np2 = 1;
  while (np2 < N) np2 <<= 1;
  const int L = np2 < 32 ? 32 / np2 : 1;        // lanes per expert column
  const int CPL = np2 > 32 ? np2 / 32 : 1;      // expert columns per lane
  const int part = np2 < 32 ? lane / np2 : 0;
  const int R = (nblk + L - 1) / L;             // <= MAXR
  const int r0 = min(nblk, part * R), r1 = min(nblk, r0 + R);
  const long long C = a.C;
  float fp = 0.f;  // sum over this lane's experts of count * sum of P
  for (int cc = 0; cc < CPL; ++cc) {
    const int col = np2 < 32 ? lane % np2 : lane + 32 * cc;
    const bool mine = col < N;
    int c[MAXR];
    float p[MAXR];
#pragma unroll
    for (int u = 0; u < MAXR; ++u) {
      const bool in = mine && r0 + u < r1;
      c[u] = in ? a.blk_counts[(size_t)(r0 + u) * N + col] : 0;
      p[u] = in ? a.blk_psum[(size_t)(r0 + u) * N + col] : 0.f;
    }
    int isum = 0;
    float fsum = 0.f;
#pragma unroll
    for (int u = 0; u < MAXR; ++u) {
      isum += c[u];
      fsum += p[u];
    }
    int before = 0, total = isum;  // the column's slots in earlier ranges, and in all
    float ftot = fsum;
    if (L > 1) {
      const int base_lane = lane % np2;
      total = 0;
      ftot = 0.f;
      for (int q = 0; q < L; ++q) {
        const int v = __shfl_sync(FULL, isum, base_lane + q * np2);
        const float fv = __shfl_sync(FULL, fsum, base_lane + q * np2);
        if (q < part) before += v;
        total += v;
        ftot += fv;
      }
    }
    if (mine) {  // exclusive per-expert base of every block
      int run = before;
#pragma unroll
      for (int u = 0; u < MAXR; ++u) {
        if (r0 + u < r1) a.blk_counts[(size_t)(r0 + u) * N + col] = run;
        run += c[u];
      }
    }
    const int kept = (C < 0 || (long long)total <= C) ? total : (int)C;
    if (mine && part == 0) {
      s_rows[col] = kept;
      a.counts[col] = total;
      a.kept[col] = kept;
      if (a.user_counts != nullptr) a.user_counts[col] = total;
      if (a.user_kept != nullptr) a.user_kept[col] = kept;
      fp = fmaf((float)total, ftot, fp);
    }
  }
  for (int j = lane; j < a.S; j += 32) {  // shared experts take every token
    s_rows[N + j] = a.T;
    a.counts[N + j] = a.T;
    a.kept[N + j] = a.T;
  }
  // aux = N * sum_e (counts_e / (T*k)) * (Psum_e / T), as in finish_routing
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) fp += __shfl_xor_sync(FULL, fp, d);
  if (lane == 0) {
    *a.cap = (int32_t)C;
    const float Tf = (float)a.T;
    *a.aux = a.T > 0 ? (float)N * (fp / (Tf * (float)a.k)) / Tf : 0.f;
  }
  __syncwarp();
  ExpertLayout lay;
  lay.offsets = a.offsets;
  for (int tb = 0; tb < 2; ++tb) {
    lay.tile_first[tb] = a.tile_first[tb];
    lay.num_mtiles[tb] = a.num_mtiles[tb];
  }
  layout_experts(s_rows, Ntot, lay);
}

}  // namespace route
}  // namespace moe
