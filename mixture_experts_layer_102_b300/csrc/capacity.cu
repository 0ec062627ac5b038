// Dispatch of the MoE layer: every slot's final rank among its expert's slots (the
// in-block rank plus the block's per-expert base from the routing decisions), the
// capacity decision, and the gather of x into the expert-contiguous buffer.
//
// Each expert keeps its first C routed slots in token order and the rest are dropped
// to the residual (cf-1.com/news/5914943 section 2.3 note; 2kiu.com/news/2885792
// section 3.1 keeps each expert's earliest tokens up to its capacity, section 2.2 capacity
// factor). Kept slots go to row offsets[e] + rank of the permuted buffer ("scatter
// tokens into expert queues", devpress.csdn.net MoE page section 4.1), copied with
// 16-byte vectors, one warp per token.
//
// With overflow rerouting, a dropped slot whose proposal its new expert accepted goes
// to that expert's rows after the expert's own count, and its index entry becomes
// the new expert.
//
// Shared experts (hotelren.com/news/5904824 section 3.3) are slots k..k+S-1 of every
// valid token: row offsets[N+j] + the token's rank among the valid tokens. A padding
// token (index -1 from the routing decisions) gets no row and every slot dropped.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int MAX_SLOTS = 32 + MAX_SHARED;

// One warp per token; a block is 8 tokens.
template <typename TIn, bool COPY>
__global__ void __launch_bounds__(256) dispatch_kernel(DispatchArgs a) {
  __shared__ int32_t rows[8][MAX_SLOTS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  // The token's first VPL x vectors per lane are requested before the wait (x is the
  // caller's input) and before the chain of dependent index loads below.
  constexpr int VPL = 8;
  const bool live = t < a.T;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const TIn*>(a.x) +
                                                    (size_t)(live ? t : 0) * a.H);
  const int nvec = a.H * (int)sizeof(TIn) / 16;
  uint4 val[VPL];
  if (COPY && live) {
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      const int v = u * 32 + lane;
      if (v < nvec) val[u] = src[v];
    }
  }
  pdl_wait();  // ranks, bases and offsets come from the routing-decision kernel
  pdl_trigger();
  if (!live) return;
  const int slots = a.k + a.S;
  const long long C = a.valid != nullptr ? (long long)*a.cap : a.C;
  const int blk = t / a.tokens_per_block;
  for (int sl = lane; sl < slots; sl += 32) {
    int row = -1;
    if (sl < a.k) {  // routed slot
      const int j = t * a.k + sl;
      const int e = a.idx[j];
      if (e < 0 && a.valid != nullptr && a.valid[t] == 0) {
        a.drop[j] = 1;  // padding token
      } else if (e < 0 || e >= a.N) {
        report(a.status, STATUS_BAD_INDEX);
        a.drop[j] = 1;
      } else {
        // base, in-block rank and offset are independent loads: one round trip
        const int base = a.blk_base[(size_t)blk * a.N + e];
        const int srank = a.slot_rank[j];
        const int off = a.offsets[e];
        const long long rank = (long long)base + srank;
        bool kept = C < 0 || rank < C;
        if (kept) {
          row = off + (int)rank;
        } else if (a.rr_exp != nullptr) {  // rerouted: after the new expert's own rows
          const int c = a.rr_exp[j];
          if (c >= 0 && c < a.N) {
            const long long r2 = (long long)a.rr_base[(size_t)blk * a.N + c] + a.rr_rank[j];
            const long long own = a.counts[c];  // < C: the expert had room
            if (r2 < C - own) {
              kept = true;
              row = a.offsets[c] + (int)(own + r2);
              a.idx[j] = c;
            }
          }
        }
        a.drop[j] = kept ? 0 : 1;
      }
    } else if (a.valid == nullptr || a.valid[t] != 0) {  // shared expert N + (sl - k)
      const int vr = a.valid == nullptr ? t : a.blk_vbase[blk] + a.vrank[t];
      row = a.offsets[a.N + sl - a.k] + vr;
    }
    if (row >= a.A_cap) {
      report(a.status, STATUS_BAD_INDEX);
      row = -1;
    }
    if (row >= 0) a.row_token[row] = t;
    a.slot_row[(size_t)t * slots + sl] = row;
    rows[warp][sl] = row;
  }
  __syncwarp();
  if (COPY) {
    uint4* dst = reinterpret_cast<uint4*>(a.xp);
    for (int v0 = 0; v0 < nvec; v0 += 32 * VPL) {
      if (v0 > 0) {
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) val[u] = src[v];
        }
      }
      for (int s = 0; s < slots; ++s) {
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
