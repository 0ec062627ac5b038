// Capacity and dispatch of the MoE layer.
//
// Each expert keeps its first C routed slots in token order and the rest are dropped
// to the residual (cf-1.com/news/5914943 section 2.3 note; 2kiu.com/news/2885792
// section 3.1 keeps "the first capacity tokens" per expert, section 2.2 capacity
// factor). Flattening the slots as j = t*k + s keeps token order per expert (a token
// picks an expert at most once), so the rank of slot j is the number of earlier
// slots with the same expert: a stable counting-sort rank, computed without atomics
// so that the kept set never depends on scheduling.
//
//   capacity_count_kernel  per block of 1024 slots: per-expert counts and each slot's
//                          rank inside the block (warp match + per-warp prefix)
//   capacity_scan_kernel   one block: per-expert exclusive scan over blocks, totals,
//                          kept = min(count, C), expert offsets, the GEMM row-tile
//                          table and aux = N * sum_e f_e * P_e
//   dispatch_kernel        per token: final rank, drop mask, permuted row, and the
//                          gather of x into the expert-contiguous buffer (16-byte
//                          vectors; "scatter tokens into expert queues",
//                          devpress.csdn.net MoE page section 4.1)
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(1024)
capacity_count_kernel(const int32_t* __restrict__ idx, int A, int N,
                      int32_t* __restrict__ chunk_counts, int32_t* __restrict__ slot_rank,
                      uint32_t* status) {
  extern __shared__ int32_t wc[];  // [32 warps][N]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 32 * N; i += 1024) wc[i] = 0;
  __syncthreads();
  const int j = blockIdx.x * COUNT_CHUNK + tid;
  int e = -1;
  if (j < A) {
    e = idx[j];
    if (e < 0 || e >= N) {
      report(status, STATUS_BAD_INDEX);
      e = -1;
    }
  }
  const uint32_t peers = __match_any_sync(0xffffffffu, e);
  const int r = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && r == 0) wc[warp * N + e] = __popc(peers);
  __syncthreads();
  for (int c = tid; c < N; c += 1024) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = wc[w * N + c];
      wc[w * N + c] = run;
      run += v;
    }
    chunk_counts[(size_t)blockIdx.x * N + c] = run;
  }
  __syncthreads();
  if (e >= 0) slot_rank[j] = wc[warp * N + e] + r;
}

// One block of 1024 threads. G = 1024 / pow2ceil(N) threads share an expert column.
__global__ void __launch_bounds__(1024) capacity_scan_kernel(ScanArgs a) {
  __shared__ int32_t ipart[1024];
  __shared__ float fpart[1024];
  __shared__ int32_t s_counts[256], s_kept[256], s_off[257], s_tile0[257];
  __shared__ float s_psum[256];
  const int tid = threadIdx.x;
  const int N = a.N;
  int np2 = 1;
  while (np2 < N) np2 <<= 1;
  const int G = 1024 / np2;
  const int col = tid / G, g = tid - col * G;

  const int R = (a.nchunks + G - 1) / G;
  const int r0 = min(a.nchunks, g * R), r1 = min(a.nchunks, r0 + R);
  const int Rp = (a.npsum + G - 1) / G;
  const int p0 = min(a.npsum, g * Rp), p1 = min(a.npsum, p0 + Rp);
  int isum = 0;
  float fsum = 0.f;
  if (col < N) {
#pragma unroll 4
    for (int r = r0; r < r1; ++r) isum += a.chunk_counts[(size_t)r * N + col];
#pragma unroll 4
    for (int r = p0; r < p1; ++r) fsum += a.psum_part[(size_t)r * N + col];
  }
  ipart[tid] = isum;
  fpart[tid] = fsum;
  __syncthreads();
  if (col < N && g == 0) {
    int run = 0;
    float p = 0.f;
    for (int q = 0; q < G; ++q) {
      const int v = ipart[tid + q];
      ipart[tid + q] = run;
      run += v;
      p += fpart[tid + q];
    }
    const int kept = (a.C < 0 || (long long)run <= a.C) ? run : (int)a.C;
    s_counts[col] = run;
    s_kept[col] = kept;
    s_psum[col] = p;
    a.counts[col] = run;
    a.kept[col] = kept;
    if (a.user_counts != nullptr) a.user_counts[col] = run;
    if (a.user_kept != nullptr) a.user_kept[col] = kept;
  }
  __syncthreads();
  if (col < N) {  // exclusive per-expert base of every count block
    int run = ipart[tid];
    for (int r = r0; r < r1; ++r) {
      const int v = a.chunk_counts[(size_t)r * N + col];
      a.chunk_counts[(size_t)r * N + col] = run;
      run += v;
    }
  }
  if (tid == 0) {
    int off = 0, tiles = 0;
    float fp = 0.f;
    for (int e = 0; e < N; ++e) {
      s_off[e] = off;
      s_tile0[e] = tiles;
      a.offsets[e] = off;
      off += s_kept[e];
      tiles += (s_kept[e] + GEMM_BM - 1) / GEMM_BM;
      fp = fmaf((float)s_counts[e], s_psum[e], fp);
    }
    s_off[N] = off;
    s_tile0[N] = tiles;
    a.offsets[N] = off;
    *a.num_mtiles = tiles;
    // aux = N * sum_e (counts_e / (T*k)) * (Psum_e / T)
    // (counts <= T*k and sum_e P_e = T keep every term well inside fp32 range)
    const float Tf = (float)a.T;
    *a.aux = a.T > 0 ? (float)N * (fp / (Tf * (float)a.k)) / Tf : 0.f;
  }
  __syncthreads();
  const int total = s_tile0[N];
  for (int i = tid; i < total; i += 1024) {
    int lo = 0, hi = N - 1;  // last expert with s_tile0[e] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tile0[mid] <= i) lo = mid; else hi = mid - 1;
    }
    a.tile_expert[i] = lo;
    a.tile_row0[i] = s_off[lo] + (i - s_tile0[lo]) * GEMM_BM;
  }
}

// One warp per token; a block is 8 tokens.
template <typename TIn, bool COPY>
__global__ void __launch_bounds__(256) dispatch_kernel(DispatchArgs a) {
  __shared__ int32_t rows[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.T) return;
  int row = -1;
  if (lane < a.k) {
    const int j = t * a.k + lane;
    const int e = a.idx[j];
    if (e < 0 || e >= a.N) {
      report(a.status, STATUS_BAD_INDEX);
      a.drop[j] = 1;
    } else {
      const long long rank =
          (long long)a.chunk_base[(size_t)(j / COUNT_CHUNK) * a.N + e] + a.slot_rank[j];
      const bool kept = a.C < 0 || rank < a.C;
      if (kept) {
        row = a.offsets[e] + (int)rank;
        if (row >= a.A_cap) {
          report(a.status, STATUS_BAD_INDEX);
          row = -1;
        } else {
          a.row_token[row] = t;
        }
      }
      a.drop[j] = kept ? 0 : 1;
    }
    a.slot_row[j] = row;
    rows[warp][lane] = row;
  }
  __syncwarp();
  if (COPY) {
    const TIn* src = static_cast<const TIn*>(a.x) + (size_t)t * a.H;
    TIn* dst = static_cast<TIn*>(a.xp);
    constexpr int EPV = 16 / sizeof(TIn);  // elements per 16-byte vector
    const int nvec = a.H / EPV;
    for (int v = lane; v < nvec; v += 32) {
      const uint4 val = reinterpret_cast<const uint4*>(src)[v];
      for (int s = 0; s < a.k; ++s) {
        const int r = rows[warp][s];
        if (r >= 0) reinterpret_cast<uint4*>(dst + (size_t)r * a.H)[v] = val;
      }
    }
  }
}

}  // namespace

cudaError_t launch_capacity_count(const int32_t* idx, int A, int N, int32_t* chunk_counts,
                                  int32_t* slot_rank, uint32_t* status, cudaStream_t stream) {
  if (A == 0) return cudaSuccess;
  const int blocks = (A + COUNT_CHUNK - 1) / COUNT_CHUNK;
  capacity_count_kernel<<<blocks, COUNT_CHUNK, 32 * N * sizeof(int32_t), stream>>>(
      idx, A, N, chunk_counts, slot_rank, status);
  return cudaGetLastError();
}

cudaError_t launch_capacity_scan(const ScanArgs& a, cudaStream_t stream) {
  capacity_scan_kernel<<<1, 1024, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dispatch(int dtype, bool copy, const DispatchArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int blocks = (a.T + 7) / 8;
  if (dtype == 1) {
    if (copy) dispatch_kernel<__nv_bfloat16, true><<<blocks, 256, 0, stream>>>(a);
    else dispatch_kernel<__nv_bfloat16, false><<<blocks, 256, 0, stream>>>(a);
  } else {
    if (copy) dispatch_kernel<float, true><<<blocks, 256, 0, stream>>>(a);
    else dispatch_kernel<float, false><<<blocks, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace moe
