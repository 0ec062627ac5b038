// Routing decisions of the MoE layer in one launch: softmax, top-k and gate weights
// per token, the load-balancing statistics and aux loss, and the per-expert capacity
// ranks, offsets and GEMM tile tables.
//
//   P = softmax(logits) over all N experts; idx = top-k of the logits (ties to the
//   lower expert id); w = softmax over the k selected logits
//     (cf-1.com/news/5914943 section 2.1; hotelren.com/news/3071227 section 4.1;
//      2kiu.com/news/2885792 section 5.3)
//   aux = N * sum_e (counts_e / (T*k)) * (sum_t P[t,e] / T), counts before capacity
//     (cf-1.com/news/5914943 section 2.3)
//   rank of a slot = number of earlier slots (token order) routed to its expert; the
//   first C slots of every expert are kept (2kiu.com/news/2885792 section 3.1;
//   cf-1.com/news/5914943 section 2.3 note)
//
// A block is 32 warps; warp w handles `tpw` consecutive tokens, one at a time, and
// lane l owns experts l, l+32, ... of the current token. Each warp keeps running
// per-expert counters in shared memory, which give every slot its rank among the
// block's earlier slots of the same expert (a token picks an expert at most once, so
// slots of one expert are ordered by token); a prefix over the warps turns them into
// in-block ranks. No atomics decide positions, so the kept set never depends on
// scheduling. The partial logits of the split-K router GEMM are summed in a fixed
// order and every reduction has a fixed shape, so the results are bit-reproducible.
//
// The block that finishes last (a device-wide completion counter, no waiting) scans
// the per-block counts of every expert into per-block bases, and writes the totals,
// kept = min(count, C), the expert offsets, the GEMM row-tile tables and the aux loss;
// it then resets the counter for the next call.
//
// Options. A valid-token mask (devpress.csdn.net MoE page section 5.2: capacity counts
// only the non-padding tokens) routes the valid tokens as a batch of their own: a
// padding token gets no expert (index -1, weight 0), adds nothing to the counts or the
// probability sums, and T_valid replaces T in C and in the losses; every valid token
// gets its rank among the valid tokens (per-warp counts, a prefix over the warps, and
// per-block bases from the last block). Shared experts (hotelren.com/news/5904824
// section 3.3) are appended to the expert list as experts N..N+S-1 that keep all
// T_valid tokens, so the offsets and tile tables cover them too. Two more balance
// losses: KL(uniform || f), f_e = counts_e / (T_valid*k) (hotelren.com/news/3071227
// section 4.2), and the unbiased variance of all router probabilities
// (2kiu.com/news/2885792 section 5.1), from per-block sums of (P - 1/N)^2 (the
// probabilities of a token sum to 1, so their mean is 1/N).
#include <math.h>

#include "common.cuh"
#include "expert_layout.cuh"
#include "internal.h"
#include "route_finish.cuh"

namespace moe {
namespace {

using namespace route;

constexpr int WARPS = SELECT_WARPS;  // 32
constexpr int MAX_TPW = 4;           // tokens per warp whose ranks stay in registers

// OPT: the valid-token mask or the variance loss may be in use (read at run time);
// without it those branches are compiled out of the base layer's kernel.
// WF: the finish runs in one warp (finish_routing_warp), else in the whole block.
template <bool OPT, bool WF>
__global__ void __launch_bounds__(1024) route_select_kernel(SelectArgs a) {
  extern __shared__ int32_t dyn[];
  int32_t* cnt = dyn;                                   // [WARPS][N] running counts
  float* pw = reinterpret_cast<float*>(dyn + WARPS * a.N);  // [WARPS][N] sums of P
  __shared__ int is_last;
  __shared__ int32_t s_vbase[WARPS];   // valid tokens before each warp's range
  __shared__ float s_d2[WARPS];
  __shared__ float s_bias[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N, k = a.k;
  for (int i = threadIdx.x; i < WARPS * N; i += blockDim.x) {
    cnt[i] = 0;
    pw[i] = 0.f;
  }
  // the bias is the caller's input, not a predecessor's output: read before the wait
  if (a.bias != nullptr)
    for (int i = threadIdx.x; i < N; i += blockDim.x) s_bias[i] = a.bias[i];
  pdl_wait();  // partial logits come from the router kernel
  pdl_trigger();
  const int NI = (N + 31) >> 5;  // experts per lane, <= 8
  const int tbase = (blockIdx.x * WARPS + warp) * a.tpw;
  const bool masked = OPT && a.valid != nullptr;
  if (masked) {  // valid tokens of every warp's range -> warp bases and the block count
    int nv = 0;
    for (int i0 = 0; i0 < a.tpw; i0 += 32) {
      const int t = tbase + i0 + lane;
      const bool v = i0 + lane < a.tpw && t < a.T && a.valid[t] != 0;
      nv += __popc(__ballot_sync(0xffffffffu, v));
    }
    if (lane == 0) s_vbase[warp] = nv;
  }
  if (OPT) __syncthreads();
  if (masked && warp == 0) {
    const int c = s_vbase[lane];
    int x = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    s_vbase[lane] = x - c;
    if (lane == 31) a.blk_valid[blockIdx.x] = x;
  }
  __syncthreads();
  const bool want_d2 = OPT && a.aux_std2 != nullptr;
  const float invN = 1.f / (float)N;
  float d2 = 0.f;
  int vnext = masked ? s_vbase[warp] : 0;
  // warp-local rank and expert of this lane's slot for the first MAX_TPW tokens
  int rank_i[MAX_TPW], exp_i[MAX_TPW];
  uint32_t live_bits = 0;
#pragma unroll
  for (int u = 0; u < MAX_TPW; ++u) rank_i[u] = exp_i[u] = 0;
  for (int i = 0; i < a.tpw; ++i) {
    const int t = tbase + i;
    if (t >= a.T) break;
    if (masked && a.valid[t] == 0) {  // padding: no expert, weight 0, no statistics
      if (lane < k) {
        a.idx[(size_t)t * k + lane] = -1;
        a.w[(size_t)t * k + lane] = 0.f;
      }
      continue;
    }
    if (i < MAX_TPW) live_bits |= 1u << i;
    if (masked) {
      if (a.S > 0 && lane == 0) a.vrank[t] = vnext;
      ++vnext;
    }
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = (q < NI && lane + 32 * q < N) ? 0.f : -INFINITY;
    // sum the split partials in split order; the loads of one split are independent
#pragma unroll 4
    for (int p = 0; p < a.ksplit; ++p) {
      const float* row = a.part + ((size_t)p * a.T + t) * N;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < NI && lane + 32 * q < N) v[q] += row[lane + 32 * q];
    }
    if (a.bias != nullptr) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < NI && lane + 32 * q < N) v[q] += s_bias[lane + 32 * q];
    }
    // softmax over all N experts
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < 8; ++q) m = fmaxf(m, v[q]);
    m = warp_max(m);
    float ex[8], sum = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane + 32 * q;
      ex[q] = (q < NI && e < N) ? expf(v[q] - m) : 0.f;
      sum += ex[q];
    }
    sum = warp_sum(sum);
    const float inv = 1.f / sum;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane + 32 * q;
      if (q < NI && e < N) {
        const float pe = ex[q] * inv;
        pw[warp * N + e] += pe;
        if (want_d2) d2 = fmaf(pe - invN, pe - invN, d2);
      }
    }
    // top-k: k rounds of a warp arg-max on (logit desc, expert id asc)
    uint32_t taken = 0;
    float my_l = 0.f, l0 = 0.f;
    int my_i = 0;
    for (int s = 0; s < k; ++s) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = lane + 32 * q;
        if (q < NI && e < N && !((taken >> q) & 1u) && v[q] > bv) {  // e ascends with q
          bv = v[q];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (s == 0) l0 = bv;
      if (lane == s) {
        my_l = bv;
        my_i = bi;
      }
    }
    // gate weights (softmax over the k selected logits) and warp-local ranks; the k
    // experts of a token are distinct, so the lanes update distinct counters
    const float z = (lane < k) ? expf(my_l - l0) : 0.f;
    const float zs = warp_sum(z);
    if (lane < k) {
      const size_t j = (size_t)t * k + lane;
      a.idx[j] = my_i;
      a.w[j] = z / zs;
      const int r = cnt[warp * N + my_i]++;
      if (i < MAX_TPW) {
#pragma unroll
        for (int u = 0; u < MAX_TPW; ++u)
          if (u == i) {
            rank_i[u] = r;
            exp_i[u] = my_i;
          }
      } else {
        a.slot_rank[j] = r;
      }
    }
    __syncwarp();
  }
  if (want_d2) {
    d2 = warp_sum(d2);
    if (lane == 0) s_d2[warp] = d2;
  }
  __syncthreads();
  // exclusive prefix of the counters over the warps: the block's per-expert offsets
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    int run = 0;
    float ps = 0.f;
    for (int w = 0; w < WARPS; ++w) {
      const int c = cnt[w * N + e];
      cnt[w * N + e] = run;
      run += c;
      ps += pw[w * N + e];
    }
    a.blk_counts[(size_t)blockIdx.x * N + e] = run;
    a.blk_psum[(size_t)blockIdx.x * N + e] = ps;
  }
  if (want_d2 && threadIdx.x == 0) {
    float s2 = 0.f;
    for (int w = 0; w < WARPS; ++w) s2 += s_d2[w];
    a.blk_d2[blockIdx.x] = s2;
  }
  __syncthreads();
  for (int i = 0; i < a.tpw; ++i) {  // warp-local ranks -> in-block ranks
    const int t = tbase + i;
    if (t >= a.T) break;
    if (lane < k) {
      const size_t j = (size_t)t * k + lane;
      if (i < MAX_TPW) {
        if (!OPT || ((live_bits >> i) & 1u)) {
#pragma unroll
          for (int u = 0; u < MAX_TPW; ++u)  // static indexing keeps the arrays in registers
            if (u == i) a.slot_rank[j] = rank_i[u] + cnt[warp * N + exp_i[u]];
        }
      } else {
        const int e = a.idx[j];
        if (!OPT || e >= 0) a.slot_rank[j] += cnt[warp * N + e];
      }
    }
  }
  // The last block to get here finishes the layer-wide statistics.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if constexpr (WF) {
    if (threadIdx.x < 32) finish_routing_warp<SELECT_WARP_FINISH_ROWS>(a, gridDim.x);
  } else {
    finish_routing(a, gridDim.x);
  }
  if (threadIdx.x == 0) *a.done = 0u;  // ready for the next call
}

}  // namespace

cudaError_t launch_route_select(const SelectArgs& a, int nblk, cudaStream_t stream, bool pdl) {
  if (a.T == 0) return cudaSuccess;
  const size_t smem = (size_t)WARPS * a.N * 8;  // counters and P sums of every warp
  const bool opt = a.valid != nullptr || a.aux_std2 != nullptr;
  const bool plain = !opt && a.aux_kl == nullptr;  // the one-warp finish computes no KL
  auto kernel = opt ? route_select_kernel<true, false>
                : warp_finish_fits(a.N, nblk, plain, SELECT_WARP_FINISH_ROWS)
                    ? route_select_kernel<false, true>
                    : route_select_kernel<false, false>;
  const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kernel, dim3(nblk), dim3(WARPS * 32), smem, stream, pdl, a);
}

}  // namespace moe
