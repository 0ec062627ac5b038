// Launchers of the MoE forward kernels, called by the C-ABI layer (moe_abi.cu).
// Every launcher enqueues on `stream` and returns the launch status; `pdl` launches
// the (first) kernel as a programmatic dependent of the previous kernel of the stream.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Tile and block geometry shared between the host plan and the kernels.
constexpr int ROUTER_TOKENS = 64;      // tokens per router-logits block
constexpr int ROUTER_KC = 32;          // hidden columns per router k-chunk
constexpr int SELECT_WARPS = 32;       // warps per routing-decision block
constexpr int TILE_ROWS_1 = 128;       // rows per expert GEMM tile on one CTA
constexpr int TILE_ROWS_2 = 256;       // rows per expert GEMM tile on a CTA pair

// ---------------------------------------------------------------- router
// Partial logits part[split][t][e] = sum over this split's hidden columns of
// x[t,h] * w_router[h,e]. dtype: 0 f32, 1 bf16.
cudaError_t launch_router_logits(int dtype, const void* x, const void* w_router, float* part,
                                 int T, int H, int N, int ksplit, int chunks_per_split,
                                 cudaStream_t stream);

// bf16 router logits on tcgen05: W_r is first copied K-major into wrt [N_pad, H]
// (N_pad = router_tc_npad(N)); partials as above with the split from router_tc_split.
int router_tc_npad(int N);
void router_tc_split(int T, int H, int* ksplit, int* kc_per_split);
cudaError_t launch_router_logits_tc(const void* x, const void* w_router, void* wrt, float* part,
                                    int T, int H, int N, uint32_t* status, cudaStream_t stream,
                                    bool pdl);

// ---------------------------------------------------------------- routing decisions
struct SelectArgs {
  const float* part;            // [ksplit][T][N] partial logits
  int ksplit;
  const float* bias;            // [N] or null
  int T, N, k;
  int tpw;                      // tokens per warp; a block is SELECT_WARPS warps
  int32_t* idx;                 // [T*k] top-k experts
  float* w;                     // [T*k] gate weights
  int32_t* slot_rank;           // [T*k] rank among the block's slots of the expert
  int32_t* blk_counts;          // [nblk][N] counts, then exclusive per-expert bases
  float* blk_psum;              // [nblk][N] sums of P
  unsigned* done;               // completion counter, zero between calls
  long long C;                  // capacity, < 0 for no limit
  int32_t* counts;              // [N] slots per expert before capacity
  int32_t* kept;                // [N] after capacity
  int32_t* offsets;             // [N+1] first permuted row of each expert
  // GEMM row-tile tables for 128-row tiles [0] and 256-row tiles [1]: expert and
  // first permuted row of each tile, and the number of tiles
  int32_t* tile_expert[2];
  int32_t* tile_row0[2];
  int32_t* num_mtiles[2];
  int32_t* tile_first[2];       // [N+1] first tile of each expert (and the total)
  float* aux;                   // [1]
  int32_t* user_counts;         // optional copies for the caller
  int32_t* user_kept;
};
// Softmax, top-k and gate weights, capacity ranks, and (in the block that finishes
// last) the per-expert scan, offsets, tile tables and aux loss.
cudaError_t launch_route_select(const SelectArgs& a, int nblk, cudaStream_t stream, bool pdl);

// ---------------------------------------------------------------- dispatch
struct DispatchArgs {
  const int32_t* idx;           // [T*k]
  const int32_t* slot_rank;     // [T*k] rank within its routing-decision block
  const int32_t* blk_base;      // [nblk][N] per-expert base of every such block
  int tokens_per_block;
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
cudaError_t launch_dispatch(int dtype, bool copy, const DispatchArgs& a, cudaStream_t stream,
                            bool pdl);

// ---------------------------------------------------------------- experts
struct GroupedGemmArgs {
  const void* A;                // [A_cap, K] permuted rows (xp or h)
  int A_rows;                   // A_cap
  const void* B0;               // [N, n_cols, K] (W1 or W2)
  const void* B1;               // [N, n_cols, K] (W3) or null
  void* out;                    // [A_cap, n_cols]
  int K, n_cols, N;
  bool swiglu;                  // out = silu(A B0^T) * (A B1^T), else A B0^T
  bool pair;                    // 256-row tiles on CTA pairs (else 128-row tiles)
  const int32_t* tile_expert;   // the table that matches the tile shape
  const int32_t* tile_row0;
  const int32_t* offsets;
  const int32_t* num_mtiles;
  const int32_t* tile_first;    // [N+1] first tile of each expert in that table
  int max_mtiles;
  uint32_t* status;
};
// float32 CUDA-core path (exact fp32 FMA, no TF32).
cudaError_t launch_grouped_gemm_simt(const GroupedGemmArgs& a, cudaStream_t stream);
// bf16 tcgen05 tensor-core path (TMA-fed, TMEM accumulators), sm_103a.
cudaError_t launch_grouped_gemm_tc(const GroupedGemmArgs& a, cudaStream_t stream, bool pdl);

// ---------------------------------------------------------------- combine
cudaError_t launch_combine(int dtype, const void* ye, const int32_t* slot_row, const float* w,
                           int T, int k, int H, void* out, cudaStream_t stream, bool pdl);

}  // namespace moe
