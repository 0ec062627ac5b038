// Router GEMM and routing decisions of bf16 layers in one launch.
//
//   logits = x W_r^T (+ b)      the router's linear layer (cf-1.com/news/5914943 section
//                               2.1; 2kiu.com/news/2885792 section 3.1)
//   P = softmax(logits); idx = top-k of the logits, ties to the lower expert id; w =
//   softmax over the k selected logits (cf-1.com/news/5914943 section 2.1;
//   hotelren.com/news/3071227 section 4.1; 2kiu.com/news/2885792 section 5.3)
//   counts, sums of P, capacity ranks in token order, offsets and the aux loss as in
//   the routing-decision kernel (route_select.cu), whose outputs this kernel writes in
//   the same form with a block of 128 tokens.
//
// One CTA per 128-token tile, 256 threads (512 above 32 experts), no split of K, so
// the logits never leave the CTA as partial sums:
//   warp 0      TMA producer: x rows and W_r ([N, H], N_pad = N rounded up to 16 rows,
//               zero past N) stream through as many 128-byte-swizzled stages as shared
//               memory holds, so the load pipeline covers HBM latency.
//   warp 1      TMEM allocator; one thread issues tcgen05.mma.cta_group::1 (M=128,
//               N=N_pad, K=16) into a TMEM accumulator.
//   warps 2-5   read the accumulator back (one token per thread: the TMEM lane) and
//               stage the logits (+ bias) in the freed stage memory.
//   all warps   two (four) threads per token (experts e = h mod 2 (4) each, combined by
//               shuffles) make the token's decisions: softmax by max and sum, the top k
//               by k passes, each taking the best logit strictly after the previous
//               pick in the order (logit descending, id ascending), the gate weights,
//               and the token's row of probabilities.
//   all warps   per expert, in a fixed order over the tile's rows: the sum of P, the
//               count, and each slot's rank among the tile's earlier slots of that
//               expert (its rank in token order inside the tile).
// The CTA that finishes last (a completion counter, no waiting) runs the same finish
// as the routing-decision kernel: per-block bases, capacity, losses, expert layout.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "route_finish.cuh"
#include "tc_util.cuh"

namespace moe {
namespace {

using namespace tc;
using namespace route;

constexpr int BK = 64;                          // 64 bf16 = one 128-byte swizzle row
constexpr int TOK = 128;                        // tokens per CTA (TMEM lanes)
constexpr uint32_t A_BYTES = TOK * BK * 2;      // 16 KB
constexpr int MAX_STAGES = 16;

// Row stride (floats) of the tile's logits in shared memory: at least N + 1 and an odd
// multiple of tpt (the threads per token), so the tpt threads of each of a warp's
// 32/tpt tokens (experts e = h mod tpt each) fall in 32 different banks.
__host__ __device__ constexpr int logit_stride(int N, int tpt) {
  return ((N + 1 + tpt - 1) / tpt) % 2 == 1 ? (N + 1 + tpt - 1) / tpt * tpt
                                             : ((N + 1 + tpt - 1) / tpt + 1) * tpt;
}

struct FusedArgs {
  SelectArgs s;        // outputs, options and workspace arrays of the routing decisions
  float* logits;       // [T][N] logits with bias, for the rerouting kernel, or null
  int kc_total;        // H / 64
  int n_pad, stages;
  uint32_t idesc, tmem_cols, b_bytes, stage_bytes, region_bytes;
  uint32_t* status;
};

// WF: the finish runs in one warp (finish_routing_warp), else in the whole CTA.
// NUM_THREADS: 256 (two threads per token in the decisions) or 512 (four).
template <bool WF, int NUM_THREADS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
route_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   FusedArgs f) {
  constexpr int TPT = NUM_THREADS / TOK;  // threads per token in the decisions
  const SelectArgs& a = f.s;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int STAGES = f.stages;
  const uint32_t full_bar = base + f.region_bytes;
  const uint32_t empty_bar = full_bar + 8 * MAX_STAGES;
  const uint32_t accf_bar = empty_bar + 8 * MAX_STAGES;
  int* misc = reinterpret_cast<int*>(base_ptr + f.region_bytes + 8 * (2 * MAX_STAGES + 1));
  volatile int* abort_flag = misc + 1;
  __shared__ float s_bias[256];
  __shared__ uint8_t s_valid[TOK];
  __shared__ int is_last;
  __shared__ double s_dd[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N, k = a.k;
  const int m0 = blockIdx.x * TOK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar + 8 * s, 1);
      mbar_init(empty_bar + 8 * s, 1);
    }
    mbar_init(accf_bar, 1);
    misc[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&tmX);
    prefetch_map(&tmW);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(misc)),
                 "r"(f.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // the bias is the caller's input, not a predecessor's output: read before the wait
  for (int i = threadIdx.x; i < N; i += NUM_THREADS)
    s_bias[i] = a.bias != nullptr ? a.bias[i] : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  pdl_wait();  // x and W_r may come from the caller's previous kernel on the stream
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------- TMA producer
      int stage = 0;
      uint32_t phase = 0, used = 0, last_parity = 0;
      bool ok = true;
      for (int kc = 0; kc < f.kc_total; ++kc) {
        if (!mbar_wait(empty_bar + 8 * stage, phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const uint32_t sA = base + stage * f.stage_bytes;
        const uint32_t fb = full_bar + 8 * stage;
        mbar_expect_tx(fb, A_BYTES + f.b_bytes);
        tma_load_2d<1>(sA, &tmX, fb, kc * BK, m0);
        tma_load_2d<1>(sA + A_BYTES, &tmW, fb, kc * BK, 0);
        used |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        report(f.status, STATUS_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      for (int s = 0; s < STAGES; ++s)
        if ((used >> s) & 1u)
          mbar_wait(full_bar + 8 * s, (last_parity >> s) & 1u, nullptr, DRAIN_LIMIT_NS);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kc = 0; kc < f.kc_total; ++kc) {
        if (!mbar_wait(full_bar + 8 * stage, phase, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sA = base + stage * f.stage_bytes;
        const uint64_t da = sw128_desc(sA);
        const uint64_t db = sw128_desc(sA + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma<1>(tmem, da + 2 * kk, db + 2 * kk, f.idesc, (kc > 0 || kk > 0) ? 1u : 0u);
        tc_commit<1>(empty_bar + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        report(f.status, STATUS_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      tc_commit<1>(accf_bar);  // also drains: every MMA above is complete when it flips
    }
  }
  // Epilogue shared memory, in the stage region (every load has landed and every MMA
  // has read its operands once the accumulator barrier flips):
  //   L  [TOK][LS]  logits, then probabilities     (fp32, LS = logit_stride(N, TPT))
  //   SEL[TOK][k]   the selected experts            (int32)
  //   CH [TOK][N]   slot + 1 of a selected expert   (bytes, 0 = not selected)
  const int LS = logit_stride(N, TPT);
  float* L = reinterpret_cast<float*>(base_ptr);
  int32_t* SEL = reinterpret_cast<int32_t*>(base_ptr + (size_t)TOK * LS * 4);
  uint8_t* CH = base_ptr + (size_t)TOK * LS * 4 + (size_t)TOK * k * 4;
  if (warp >= 2 && warp < 6) {  // ------------------------------- accumulator -> smem
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int t = m0 + r;
    bool ok = mbar_wait(accf_bar, 0, abort_flag, WAIT_LIMIT_NS);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
      for (int c = 0; c < f.n_pad; c += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + c, v);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int e = c + q;
          if (e < N) {
            const float l = __uint_as_float(v[q]) + s_bias[e];
            L[r * LS + e] = l;
            if (f.logits != nullptr && t < a.T) f.logits[(size_t)t * N + e] = l;
          }
        }
      }
    } else {
      if (lane == 0) {
        report(f.status, STATUS_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {  // the accumulator has been read
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(f.tmem_cols)
                 : "memory");
  }
  // ------------------------------------------------- per-token decisions (all warps)
  // TPT threads per token, adjacent lanes: thread h of token r takes the experts
  // e = h mod TPT. Every thread runs the picks and the sum (so the shuffles are never
  // divergent); only live tokens write. Any timeout (abort flag) leaves every
  // token of the tile without a decision, as padding. Passes over the token's experts:
  // k picks (the first also clears the selection marks, and its value is the row's
  // maximum), then one pass that turns each logit into exp(l - max), summing them.
  // The probabilities are those values times 1/sum, applied where they are read.
  const bool masked = a.valid != nullptr;
  const bool want_d2 = a.aux_std2 != nullptr;
  __shared__ float s_inv[TOK];  // 1/sum of each token's exponentials (0: not live)
  float d2 = 0.f;
  {
    const unsigned FULL = 0xffffffffu;
    const int r = threadIdx.x / TPT, h = threadIdx.x % TPT;
    const int t = m0 + r;
    float* row = L + r * LS;
    uint8_t* ch = CH + (size_t)r * N;
    int32_t* sel = SEL + r * k;
    const bool live = *abort_flag == 0 && t < a.T && (!masked || a.valid[t] != 0);
    if (h == 0) s_valid[r] = live ? 1 : 0;
    // top k: pick j is the best logit strictly after pick j-1 in (logit desc, id asc);
    // each thread scans its experts, and the token's threads keep the best candidate
    float pl = INFINITY, l0 = 0.f, zs = 0.f, m = -INFINITY;
    int pi = -1;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = -1;
#pragma unroll 8
      for (int e = h; e < N; e += TPT) {
        const float v = row[e];
        if (j == 0) ch[e] = 0;
        const bool after = v < pl || (v == pl && e > pi);
        if (after && (bi < 0 || v > bv)) {
          bv = v;
          bi = e;
        }
      }
#pragma unroll
      for (int o = 1; o < TPT; o <<= 1) {  // the token's threads keep the best candidate
        const float ov = __shfl_xor_sync(FULL, bv, o);
        const int oi = __shfl_xor_sync(FULL, bi, o);
        if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if (j == 0 && bi >= 0) m = bv;  // the largest logit of the row
      if (bi < 0) {  // only NaN logits leave no candidate: keep the index in range
        bi = j;
        bv = row[j];
      }
      if (j % TPT == h) sel[j] = bi;
      if (j == 0) l0 = bv;
      zs += expf(bv - l0);
      pl = bv;
      pi = bi;
    }
    __syncwarp();  // the token's picks and cleared marks are in place
    if (live) {
      for (int j = h; j < k; j += TPT) {  // gate weights: softmax over the k selected logits
        const int e = sel[j];
        a.idx[(size_t)t * k + j] = e;
        a.w[(size_t)t * k + j] = expf(row[e] - l0) / zs;
        ch[e] = (uint8_t)(j + 1);
      }
    } else if (t < a.T) {  // padding: no expert, weight 0
      for (int j = h; j < k; j += TPT) {
        a.idx[(size_t)t * k + j] = -1;
        a.w[(size_t)t * k + j] = 0.f;
      }
    }
    __syncwarp();  // the gates have read the logits they need
    float sum = 0.f;
#pragma unroll 8
    for (int e = h; e < N; e += TPT) {  // exp(l - max) replaces each logit
      const float x = live ? expf(row[e] - m) : 0.f;
      row[e] = x;
      sum += x;
    }
#pragma unroll
    for (int o = 1; o < TPT; o <<= 1) sum += __shfl_xor_sync(FULL, sum, o);  // same on all
    const float inv = 1.f / sum;
    if (h == 0) s_inv[r] = live ? inv : 0.f;
    if (want_d2 && live) {
      const float invN = 1.f / (float)N;
#pragma unroll 8
      for (int e = h; e < N; e += TPT) {
        const float pe = __fmul_rn(row[e], inv);
        d2 = fmaf(pe - invN, pe - invN, d2);
      }
    }
  }
  __syncthreads();
  // ------------------------------------------------------ per-expert column pass
  // Thread (g, e) covers rows [g*R, g*R + R) of expert e: count, sum of P; the groups'
  // counts are prefixed in order and every slot gets its rank inside the tile.
  {
    int np2 = 1;
    while (np2 < N) np2 <<= 1;
    int G = NUM_THREADS / np2;
    if (G > TOK) G = TOK;
    const int R = TOK / G;
    const int e = threadIdx.x % np2, g = threadIdx.x / np2;
    __shared__ int32_t s_gc[NUM_THREADS];
    __shared__ float s_gp[NUM_THREADS];
    int cnt = 0;
    float ps = 0.f;
    const bool mine = e < N && g < G;
    if (mine) {
      for (int r = g * R; r < g * R + R; ++r) {
        ps += __fmul_rn(L[r * LS + e], s_inv[r]);  // the token's probability of e
        cnt += CH[(size_t)r * N + e] != 0;
      }
      s_gc[g * np2 + e] = cnt;
      s_gp[g * np2 + e] = ps;
    }
    __syncthreads();
    if (mine) {
      int rank = 0;
      for (int h = 0; h < g; ++h) rank += s_gc[h * np2 + e];
      for (int r = g * R; r < g * R + R; ++r) {
        const int c = CH[(size_t)r * N + e];
        if (c != 0) a.slot_rank[(size_t)(m0 + r) * k + (c - 1)] = rank++;
      }
      if (g == G - 1) {  // this block's totals, summed over the groups in order
        int tc = 0;
        float tp = 0.f;
        for (int h = 0; h < G; ++h) {
          tc += s_gc[h * np2 + e];
          tp += s_gp[h * np2 + e];
        }
        a.blk_counts[(size_t)blockIdx.x * N + e] = tc;
        a.blk_psum[(size_t)blockIdx.x * N + e] = tp;
      }
    }
  }
  if (masked && warp == 0) {  // valid tokens of the tile: ranks and count
    int run = 0;
    for (int c = 0; c < TOK; c += 32) {
      const bool v = s_valid[c + lane] != 0;
      const uint32_t b = __ballot_sync(0xffffffffu, v);
      const int t = m0 + c + lane;
      if (v && a.S > 0) a.vrank[t] = run + __popc(b & ((1u << lane) - 1u));
      run += __popc(b);
    }
    if (lane == 0) a.blk_valid[blockIdx.x] = run;
  }
  if (want_d2) {
    const double dsum = block_sum((double)d2, s_dd);
    if (threadIdx.x == 0) a.blk_d2[blockIdx.x] = (float)dsum;
  }
  // The last CTA to get here finishes the layer-wide statistics.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if constexpr (WF) {
    if (threadIdx.x < 32) finish_routing_warp<FUSED_WARP_FINISH_ROWS>(a, gridDim.x);
  } else {
    finish_routing(a, gridDim.x);
  }
  if (threadIdx.x == 0) *a.done = 0u;  // ready for the next call
}

}  // namespace

cudaError_t launch_route_fused(const SelectArgs& s, const void* x, const void* w_router, int H,
                               float* logits, uint32_t* status, cudaStream_t stream, bool pdl) {
  if (s.T == 0) return cudaSuccess;
  FusedArgs f;
  f.s = s;
  f.logits = logits;
  f.status = status;
  f.kc_total = H / BK;
  f.n_pad = (s.N + 15) / 16 * 16;
  uint32_t cols = 32;
  while ((int)cols < f.n_pad) cols <<= 1;
  f.tmem_cols = cols;
  f.b_bytes = (uint32_t)f.n_pad * 128;
  f.stage_bytes = (A_BYTES + f.b_bytes + 1023u) & ~1023u;
  // kind::f16 descriptor: D fp32, A/B bf16, K-major, N = n_pad, M = 128
  f.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(f.n_pad >> 3) << 17) |
            ((uint32_t)(TOK >> 4) << 24);
  const int nblk = (s.T + TOK - 1) / TOK;
  // Above 32 experts the decisions and the column pass take four threads per token
  // (same-call A/B on the fine-grained layer: route stage 48.5 -> 45.1 us); the
  // smaller layers were no faster with them. With 32 or more blocks the one-warp
  // finish fits up to 16 experts.
  const bool plain = s.valid == nullptr && s.aux_kl == nullptr && s.aux_std2 == nullptr;
  const bool wf = warp_finish_fits(s.N, nblk, plain, FUSED_WARP_FINISH_ROWS);
  const int nthreads = route_fused_threads(s.N);
  const int variant = wf && nthreads == 256 ? 0 : nthreads == 512 ? 2 : 1;
  auto kernel = variant == 0 ? route_fused_kernel<true, 256>
              : variant == 1 ? route_fused_kernel<false, 256>
                             : route_fused_kernel<false, 512>;
  // the kernel's static shared memory (once per process: it does not depend on the
  // device) and the device's opt-in limit bound the dynamic part
  static size_t static_smem[3] = {0, 0, 0};
  static std::once_flag once[3];
  cudaError_t e = cudaSuccess;
  std::call_once(once[variant], [&] {
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, kernel);
    static_smem[variant] = attr.sharedSizeBytes;
  });
  const size_t kstatic = static_smem[variant];
  if (e != cudaSuccess || kstatic == 0) return e != cudaSuccess ? e : cudaErrorInvalidValue;
  size_t optin = 0;
  e = smem_optin_bytes(&optin);
  if (e != cudaSuccess) return e;
  const size_t epi = (size_t)TOK * logit_stride(s.N, nthreads / TOK) * 4 +
                     (size_t)TOK * s.k * 4 + (size_t)TOK * s.N;
  const size_t tail = 8 * (2 * MAX_STAGES + 1) + 16;  // barriers, TMEM address, abort flag
  if (optin < kstatic + 1024 + tail) return cudaErrorInvalidValue;
  const size_t avail = optin - kstatic - 1024 - tail;
  int stages = (int)(avail / f.stage_bytes);
  if (stages > MAX_STAGES) stages = MAX_STAGES;
  if (stages > f.kc_total) stages = f.kc_total > 1 ? f.kc_total : 1;
  if (stages < 1) return cudaErrorInvalidValue;
  f.stages = stages;
  size_t region = (size_t)stages * f.stage_bytes;
  if (region < epi) region = (epi + 1023) / 1024 * 1024;
  if (region > avail) return cudaErrorInvalidValue;
  f.region_bytes = (uint32_t)region;
  const size_t smem = 1024 + region + tail;
  CUtensorMap mX, mW;
  if (!make_map(&mX, x, 2, (uint64_t)H, 0, (uint64_t)s.T, TOK)) return cudaErrorInvalidValue;
  if (!make_map(&mW, w_router, 2, (uint64_t)H, 0, (uint64_t)s.N, (uint32_t)f.n_pad))
    return cudaErrorInvalidValue;
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kernel, dim3(nblk), dim3(nthreads), smem, stream, pdl, mX, mW, f);
}

}  // namespace moe
