// Overflow rerouting: one round that moves the slots capacity dropped to the next-best
// experts that still have room, instead of sending them to the residual.
//
// Sources: cf-1.com/news/5914943 section 2.3 note (overflow tokens go to other, idle
// experts); hotelren.com/news/5904824 section 3.4 and 2kiu.com/news/2885792 section
// 2.2 (overflow is dropped or routed to the next-best expert); hotelren.com/news/
// 3071227 section 4.2 (capacity-aware routing: the overloaded experts' logits are
// masked and the best remaining expert is taken).
//
// The round: an expert has room when fewer than C slots chose it (count < C). A
// token's dropped slots, in slot order, propose the token's best, second best, ...
// experts with room that it did not select (logit descending, ties to the lower id).
// Every expert accepts the proposals in token order up to its room C - count; the
// rest stay dropped. Accepted slots keep their gate weights and are placed after the
// expert's first count rows.
//
// Same block geometry as the routing decisions (32 warps, `tpw` consecutive tokens
// per warp, one at a time): a warp re-sums the logits of a token only when one of
// its slots was dropped, and ranks its proposals with per-warp counters as the
// routing decisions rank the original slots (a token proposes an expert at most
// once). The block that finishes last scans the per-block proposal counts into bases
// and writes the final rows per expert, offsets and tile tables.
#include <math.h>

#include "common.cuh"
#include "expert_layout.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int WARPS = SELECT_WARPS;

__global__ void __launch_bounds__(1024) reroute_kernel(RerouteArgs a) {
  extern __shared__ int32_t cnt[];  // [WARPS][N] proposal counters
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N, k = a.k;
  for (int i = threadIdx.x; i < WARPS * N; i += blockDim.x) cnt[i] = 0;
  pdl_wait();  // ranks, bases, counts and the capacity come from the routing decisions
  pdl_trigger();
  __syncthreads();
  const long long C = *a.cap;
  const int NI = (N + 31) >> 5;  // experts per lane, <= 8
  const int tbase = (blockIdx.x * WARPS + warp) * a.tpw;
  const int blk = blockIdx.x;
  for (int i = 0; i < a.tpw; ++i) {
    const int t = tbase + i;
    if (t >= a.T) break;
    const size_t j = (size_t)t * k + lane;
    int e = -1;
    bool dropped = false;
    if (lane < k) {
      e = a.idx[j];
      if (e >= 0 && e < N) {
        const long long r = (long long)a.blk_base[(size_t)blk * N + e] + a.slot_rank[j];
        dropped = C >= 0 && r >= C;
      }
      a.rr_exp[j] = -1;
    }
    const uint32_t lost = __ballot_sync(0xffffffffu, dropped);
    if (lost == 0) continue;
    // the token's logits for this lane's experts, summed in split order
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = 0.f;
    for (int p = 0; p < a.ksplit; ++p) {
      const float* row = a.part + ((size_t)p * a.T + t) * N;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < NI && lane + 32 * q < N) v[q] += row[lane + 32 * q];
    }
    // candidates: room left and not selected by the token
    uint32_t ok = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int ee = lane + 32 * q;
      if (q < NI && ee < N && (long long)a.counts[ee] < C) ok |= 1u << q;
      if (a.bias != nullptr && q < NI && ee < N) v[q] += a.bias[ee];
    }
    for (int s = 0; s < k; ++s) {
      const int es = __shfl_sync(0xffffffffu, e, s);
      if (es >= 0 && (es & 31) == lane) ok &= ~(1u << (es >> 5));
    }
    // the r-th dropped slot (slot order) takes the r-th best candidate
    uint32_t rest = lost;
    while (rest != 0) {
      const int s = __ffs(rest) - 1;
      rest &= rest - 1;
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int ee = lane + 32 * q;
        if (((ok >> q) & 1u) && (v[q] > bv || bi == 0x7fffffff)) {  // ee ascends with q
          bv = v[q];
          bi = ee;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi == 0x7fffffff) break;  // no candidate left
      if ((bi & 31) == lane) ok &= ~(1u << (bi >> 5));
      if (lane == s) {
        a.rr_exp[j] = bi;
        a.rr_rank[j] = cnt[warp * N + bi]++;  // warp-local rank
      }
    }
    __syncwarp();
  }
  __syncthreads();
  // exclusive prefix of the counters over the warps, and the block's proposal counts
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < WARPS; ++w) {
      const int c = cnt[w * N + e];
      cnt[w * N + e] = run;
      run += c;
    }
    a.rblk[(size_t)blk * N + e] = run;
  }
  __syncthreads();
  for (int i = 0; i < a.tpw; ++i) {  // warp-local ranks -> in-block ranks
    const int t = tbase + i;
    if (t >= a.T) break;
    if (lane < k) {
      const size_t j = (size_t)t * k + lane;
      const int c = a.rr_exp[j];
      if (c >= 0) a.rr_rank[j] += cnt[warp * N + c];
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // The last block: proposal bases per block, accepted = min(room, proposals), the
  // final rows per expert and their layout.
  __shared__ int32_t s_total[256], s_rows[MAX_EXPERTS];
  column_scan(a.rblk, gridDim.x, N, s_total);
  const int Ntot = N + a.S;
  for (int e = threadIdx.x; e < Ntot; e += blockDim.x) {
    int rows = a.kept[e];  // shared experts keep their rows
    if (e < N) {
      const long long cnt_e = a.counts[e];
      const long long room = C < 0 ? 0 : (cnt_e < C ? C - cnt_e : 0);
      const long long acc = s_total[e] < room ? s_total[e] : room;
      rows = (int)((C >= 0 && cnt_e > C ? C : cnt_e) + acc);
      a.kept[e] = rows;
      if (a.user_kept != nullptr) a.user_kept[e] = rows;
    }
    s_rows[e] = rows;
  }
  __syncthreads();
  ExpertLayout lay;
  lay.offsets = a.offsets;
  for (int tb = 0; tb < 2; ++tb) {
    lay.tile_first[tb] = a.tile_first[tb];
    lay.num_mtiles[tb] = a.num_mtiles[tb];
  }
  layout_experts(s_rows, Ntot, lay);
  if (threadIdx.x == 0) *a.done = 0u;  // ready for the next call
}

}  // namespace

cudaError_t launch_reroute(const RerouteArgs& a, int nblk, cudaStream_t stream, bool pdl) {
  if (a.T == 0) return cudaSuccess;
  const size_t smem = (size_t)WARPS * a.N * 4;
  const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(reroute_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(reroute_kernel, dim3(nblk), dim3(WARPS * 32), smem, stream, pdl, a);
}

}  // namespace moe
