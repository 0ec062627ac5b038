// Launchers of the MoE forward kernels, called by the C-ABI layer (moe_abi.cu).
// Every launcher enqueues on `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Tile and block geometry shared between the host plan and the kernels.
constexpr int ROUTER_TOKENS = 64;      // tokens per router-logits block
constexpr int ROUTER_KC = 32;          // hidden columns per router k-chunk
constexpr int COUNT_CHUNK = 1024;      // routing slots per capacity-count block
constexpr int GEMM_BM = 256;           // rows per expert GEMM tile (one CTA pair)

// ---------------------------------------------------------------- router
// Partial logits part[split][t][e] = sum over this split's hidden columns of
// x[t,h] * w_router[h,e]. dtype: 0 f32, 1 bf16.
cudaError_t launch_router_logits(int dtype, const void* x, const void* w_router, float* part,
                                 int T, int H, int N, int ksplit, int chunks_per_split,
                                 cudaStream_t stream);

// Sums the ksplit partials (+ bias), full softmax (per-block sums of P written to
// psum_part[block][e]), top-k with the lower-id tie rule and the softmax over the
// selected logits. tokens_per_warp: 1 or 8 (a block is 8 warps).
cudaError_t launch_router_select(const float* part, int ksplit, const float* bias, int T, int N,
                                 int k, int tokens_per_warp, int32_t* idx, float* w,
                                 float* psum_part, cudaStream_t stream);

// ---------------------------------------------------------------- capacity
// For each block of COUNT_CHUNK consecutive slots (slot j = t*k + s): the per-expert
// slot counts of the block and each slot's rank among the block's earlier slots of
// the same expert.
cudaError_t launch_capacity_count(const int32_t* idx, int A, int N, int32_t* chunk_counts,
                                  int32_t* slot_rank, uint32_t* status, cudaStream_t stream);

struct ScanArgs {
  int32_t* chunk_counts;        // [nchunks][N] in: counts, out: exclusive bases
  int nchunks;
  const float* psum_part;       // [npsum][N]
  int npsum;
  int T, k, N;
  long long C;                  // capacity, < 0 for no limit
  int32_t* counts;              // [N] slots per expert before capacity
  int32_t* kept;                // [N] after capacity
  int32_t* offsets;             // [N+1] first permuted row of each expert
  int32_t* tile_expert;         // [max_mtiles] expert of each GEMM row tile
  int32_t* tile_row0;           // [max_mtiles] first permuted row of each tile
  int32_t* num_mtiles;          // [1]
  float* aux;                   // [1]
  int32_t* user_counts;         // optional copies for the caller
  int32_t* user_kept;
};
cudaError_t launch_capacity_scan(const ScanArgs& a, cudaStream_t stream);

struct DispatchArgs {
  const int32_t* idx;           // [T*k]
  const int32_t* slot_rank;     // [T*k] rank within its count block
  const int32_t* chunk_base;    // [nchunks][N]
  const int32_t* offsets;       // [N+1]
  long long C;
  int T, k, N, H;
  int A_cap;                    // rows of the permuted buffer
  const void* x;                // [T,H]
  void* xp;                     // [A_cap,H] (may be null when copy is false)
  uint8_t* drop;                // [T*k]
  int32_t* slot_row;            // [T*k] permuted row of each slot, -1 when dropped
  int32_t* row_token;           // [A_cap]
  uint32_t* status;
};
cudaError_t launch_dispatch(int dtype, bool copy, const DispatchArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- experts
struct GroupedGemmArgs {
  const void* A;                // [A_cap, K] permuted rows (xp or h)
  int A_rows;                   // A_cap
  const void* B0;               // [N, n_cols, K] (W1 or W2)
  const void* B1;               // [N, n_cols, K] (W3) or null
  void* out;                    // [A_cap, n_cols]
  int K, n_cols, N;
  bool swiglu;                  // out = silu(A B0^T) * (A B1^T), else A B0^T
  const int32_t* tile_expert;
  const int32_t* tile_row0;
  const int32_t* offsets;
  const int32_t* num_mtiles;
  int max_mtiles;
  uint32_t* status;
};
// float32 CUDA-core path (exact fp32 FMA, no TF32).
cudaError_t launch_grouped_gemm_simt(const GroupedGemmArgs& a, cudaStream_t stream);
// bf16 tcgen05 tensor-core path (TMA-fed, TMEM accumulators), sm_103a.
cudaError_t launch_grouped_gemm_tc(const GroupedGemmArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- combine
cudaError_t launch_combine(int dtype, const void* ye, const int32_t* slot_row, const float* w,
                           int T, int k, int H, void* out, cudaStream_t stream);

}  // namespace moe
