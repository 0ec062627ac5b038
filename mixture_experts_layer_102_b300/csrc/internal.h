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
constexpr int MAX_SHARED = 8;          // always-on experts
constexpr int MAX_EXPERTS = 256 + MAX_SHARED;

// Expert GEMM epilogues.
enum Epilogue : int { EPI_PLAIN = 0, EPI_SWIGLU = 1, EPI_GELU = 2 };

// ---------------------------------------------------------------- router
// Partial logits part[split][t][e] = sum over this split's hidden columns of
// x[t,h] * w_router[e,h] (W_r [N,H], nn.Linear orientation). dtype: 0 f32, 1 bf16.
cudaError_t launch_router_logits(int dtype, const void* x, const void* w_router, float* part,
                                 int T, int H, int N, int ksplit, int chunks_per_split,
                                 cudaStream_t stream);

// bf16 router logits on tcgen05, partials as above with the split from
// router_tc_split; the W_r boxes are router_tc_npad(N) rows (zero past N).
int router_tc_npad(int N);
void router_tc_split(int T, int H, int* ksplit, int* kc_per_split);
cudaError_t launch_router_logits_tc(const void* x, const void* w_router, float* part, int T,
                                    int H, int N, uint32_t* status, cudaStream_t stream,
                                    bool pdl);

// ---------------------------------------------------------------- routing decisions
struct SelectArgs {
  const float* part;            // [ksplit][T][N] partial logits
  int ksplit;
  const float* bias;            // [N] or null
  int T, N, k;
  int S;                        // always-on experts N..N+S-1 (rows = the valid tokens)
  const uint8_t* valid;         // [T] 1 = real token, 0 = padding; null = all real
  int32_t* vrank;               // [T] rank of a valid token among its block's valid tokens
  int32_t* blk_valid;           // [nblk] valid tokens per block, then exclusive bases
  float* blk_d2;                // [nblk] sums of (P - 1/N)^2 (only with aux_std2)
  int32_t* cap;                 // [1] capacity of the call (-1: no limit)
  long long C;                  // capacity from T (-1: no limit), used without a mask
  double cf;                    // capacity factor (<= 0: no limit), used with a mask
  float* aux_kl;                // [1] or null: KL(uniform || f)
  float* aux_std2;              // [1] or null: unbiased variance of all P
  int tpw;                      // tokens per warp; a block is SELECT_WARPS warps
  int32_t* idx;                 // [T*k] top-k experts
  float* w;                     // [T*k] gate weights
  int32_t* slot_rank;           // [T*k] rank among the block's slots of the expert
  int32_t* blk_counts;          // [nblk][N] counts, then exclusive per-expert bases
  float* blk_psum;              // [nblk][N] sums of P
  unsigned* done;               // completion counter, zero between calls
  int32_t* counts;              // [N+S] slots per expert before capacity
  int32_t* kept;                // [N+S] after capacity
  int32_t* offsets;             // [N+S+1] first permuted row of each expert
  // GEMM row tiles of 128 rows [0] and 256 rows [1]: first tile of each expert (and
  // the total), and the number of tiles
  int32_t* num_mtiles[2];
  int32_t* tile_first[2];       // [N+S+1]
  float* aux;                   // [1]
  int32_t* user_counts;         // optional copies for the caller
  int32_t* user_kept;
};
// Softmax, top-k and gate weights, capacity ranks, and (in the block that finishes
// last) the per-expert scan, offsets, tile starts and aux loss.
cudaError_t launch_route_select(const SelectArgs& a, int nblk, cudaStream_t stream, bool pdl);

// bf16 layers: the router GEMM and the routing decisions in one launch, writing what
// launch_route_select writes with blocks of ROUTE_FUSED_TOKENS tokens (a.part, a.ksplit
// and a.tpw unused). `logits` [T][N] receives the logits with bias, or is null.
constexpr int ROUTE_FUSED_TOKENS = 128;

// The routing kernels' finish (the last block's per-expert scan, capacity, losses and
// expert layout) runs in one warp when the layer has no mask and neither optional loss
// and every lane holds its share of the per-block counts in registers: up to 32
// experts, L = 32/np2(N) lanes share an expert column and each takes at most max_rows
// block rows; above 32 experts a lane takes every block row of its columns, at most
// max_rows. The fused kernel's lanes take up to 16 rows, the routing-decision kernel's
// up to 8 (its 1024-thread blocks leave 64 registers).
constexpr int FUSED_WARP_FINISH_ROWS = 16;
constexpr int SELECT_WARP_FINISH_ROWS = 8;
inline bool warp_finish_fits(int N, int nblk, bool plain, int max_rows) {
  if (!plain) return false;
  int np2 = 1;
  while (np2 < N) np2 <<= 1;
  return np2 <= 32 ? nblk <= max_rows * (32 / np2) : nblk <= max_rows;
}
// Threads per CTA of the fused routing kernel: four threads per token in the decisions
// above 32 experts, two otherwise.
inline int route_fused_threads(int N) { return N > 32 ? 512 : 256; }
cudaError_t launch_route_fused(const SelectArgs& a, const void* x, const void* w_router, int H,
                               float* logits, uint32_t* status, cudaStream_t stream, bool pdl);

// ---------------------------------------------------------------- overflow rerouting
struct RerouteArgs {
  const float* part;            // [ksplit][T][N] partial logits
  int ksplit;
  const float* bias;            // [N] or null
  int T, N, k, S;
  int tpw;                      // the routing-decision kernel's tokens per warp
  const int32_t* idx;           // [T*k] routed experts (-1: padding)
  const int32_t* slot_rank;     // [T*k] rank within the routing-decision block
  const int32_t* blk_base;      // [nblk][N] per-expert bases of those blocks
  const int32_t* counts;        // [N] slots per expert before capacity
  int32_t* kept;                // [N+S] rows per expert: capacity's in, final out
  const int32_t* cap;           // [1] capacity of the call
  int32_t* rr_exp;              // [T*k] proposed expert of a dropped slot, -1: none
  int32_t* rr_rank;             // [T*k] rank of the proposal in its block
  int32_t* rblk;                // [nblk][N] proposals per block, then exclusive bases
  unsigned* done;               // completion counter, zero between calls
  int32_t* offsets;             // [N+S+1]
  int32_t* num_mtiles[2];
  int32_t* tile_first[2];
  int32_t* user_kept;           // [N] or null
};
// One round of rerouting of the slots that capacity dropped, and the final expert
// layout (the routing-decision kernel's block geometry).
cudaError_t launch_reroute(const RerouteArgs& a, int nblk, cudaStream_t stream, bool pdl);

// ---------------------------------------------------------------- dispatch
struct DispatchArgs {
  int32_t* idx;                 // [T*k]; a rerouted slot's entry becomes its new expert
  const int32_t* slot_rank;     // [T*k] rank within its routing-decision block
  const int32_t* blk_base;      // [nblk][N] per-expert base of every such block
  int tokens_per_block;
  const int32_t* offsets;       // [N+S+1]
  const int32_t* cap;           // [1] capacity of the call, read when a mask is given
  long long C;                  // capacity from T (-1: no limit), used without a mask
  int T, k, N, H;
  int S;                        // always-on experts
  const uint8_t* valid;         // [T] or null
  const int32_t* vrank;         // [T] valid rank inside the routing block (with a mask)
  const int32_t* blk_vbase;     // [nblk] valid tokens before each routing block
  int A_cap;                    // rows of the permuted buffer
  const void* x;                // [T,H]
  void* xp;                     // [A_cap,H] (may be null when copy is false)
  const int32_t* rr_exp;        // [T*k] rerouting proposals, or null without rerouting
  const int32_t* rr_rank;       // [T*k]
  const int32_t* rr_base;       // [nblk][N]
  const int32_t* counts;        // [N] slots per expert before capacity
  uint8_t* drop;                // [T*k]
  int32_t* slot_row;            // [T*(k+S)] permuted row of each slot, -1 when dropped
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
  int K, n_cols, N;             // N: experts in the weight tensors (routed + shared)
  int epi;                      // Epilogue: SwiGLU out = silu(A B0^T) * (A B1^T),
                                // GELU out = gelu(A B0^T), plain out = A B0^T
  bool pair;                    // 256-row tiles on CTA pairs (else 128-row tiles)
  const int32_t* offsets;       // [N+1] first permuted row of each expert (N as above)
  const int32_t* num_mtiles;    // row tiles of the tile shape
  const int32_t* tile_first;    // [N+1] first row tile of each expert in that shape
  int max_mtiles;
  uint32_t* status;
};
// float32 CUDA-core path (exact fp32 FMA, no TF32).
cudaError_t launch_grouped_gemm_simt(const GroupedGemmArgs& a, cudaStream_t stream);
// bf16 tcgen05 tensor-core path (TMA-fed, TMEM accumulators), sm_103a.
cudaError_t launch_grouped_gemm_tc(const GroupedGemmArgs& a, cudaStream_t stream, bool pdl);

// ---------------------------------------------------------------- combine
// out[t] = sum over the k routed slots of w * ye[row] plus the S shared slots with
// weight 1 (slot_row stride k+S, -1 = no row).
cudaError_t launch_combine(int dtype, const void* ye, const int32_t* slot_row, const float* w,
                           int T, int k, int S, int H, void* out, cudaStream_t stream, bool pdl);

}  // namespace moe
