// Dispatch of the MoE layer: every slot's final rank among its expert's slots (the
// in-block rank plus the block's per-expert base from the routing decisions), the
// capacity decision, and the gather of x into the expert-contiguous buffer.
//
// Each expert keeps its first C routed slots in token order and the rest are dropped
// to the residual (cf-1.com/news/5914943 section 2.3 note; 2kiu.com/news/2885792
// section 3.1 keeps "the first capacity tokens" per expert, section 2.2 capacity
// factor). Kept slots go to row offsets[e] + rank of the permuted buffer ("scatter
// tokens into expert queues", devpress.csdn.net MoE page section 4.1), copied with
// 16-byte vectors, one warp per token.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// One warp per token; a block is 8 tokens.
template <typename TIn, bool COPY>
__global__ void __launch_bounds__(256) dispatch_kernel(DispatchArgs a) {
  __shared__ int32_t rows[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  pdl_wait();  // ranks, bases and offsets come from the routing-decision kernel
  pdl_trigger();
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
          (long long)a.blk_base[(size_t)(t / a.tokens_per_block) * a.N + e] + a.slot_rank[j];
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
    // Up to VPL 16-byte loads in flight per lane before the k row stores.
    constexpr int VPL = 8;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const TIn*>(a.x) +
                                                      (size_t)t * a.H);
    uint4* dst = reinterpret_cast<uint4*>(a.xp);
    const int nvec = a.H * (int)sizeof(TIn) / 16;
    for (int v0 = 0; v0 < nvec; v0 += 32 * VPL) {
      uint4 val[VPL];
#pragma unroll
      for (int u = 0; u < VPL; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nvec) val[u] = src[v];
      }
      for (int s = 0; s < a.k; ++s) {
        const int r = rows[warp][s];
        if (r < 0) continue;
        uint4* drow = dst + (size_t)r * nvec;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) drow[v] = val[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_dispatch(int dtype, bool copy, const DispatchArgs& a, cudaStream_t stream,
                            bool pdl) {
  if (a.T == 0) return cudaSuccess;
  const dim3 grid((a.T + 7) / 8), block(256);
  if (dtype == 1)
    return copy ? launch_kernel(dispatch_kernel<__nv_bfloat16, true>, grid, block, 0, stream, pdl, a)
                : launch_kernel(dispatch_kernel<__nv_bfloat16, false>, grid, block, 0, stream, pdl,
                                a);
  return copy ? launch_kernel(dispatch_kernel<float, true>, grid, block, 0, stream, pdl, a)
              : launch_kernel(dispatch_kernel<float, false>, grid, block, 0, stream, pdl, a);
}

}  // namespace moe
