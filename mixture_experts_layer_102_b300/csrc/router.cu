// Router of the MoE layer: logits = x @ W_r (+ b), the softmax over all N experts
// (for the aux loss), top-k with ties to the lower expert id and the softmax over the
// k selected logits (cf-1.com/news/5914943 section 2.1 router pseudocode;
// hotelren.com/news/3071227 section 4.1 TopKRouter; stable tie order from
// 2kiu.com/news/2885792 section 5.3).
//
// router_logits_kernel is a split-K fp32 GEMM x W_r^T ([T,H] by W_r [N,H]) on CUDA
// cores: N <= 256
// makes it a thin product that is bound by reading x once, and the split over H keeps
// 2 blocks per SM busy when T is small (decode). The routing decisions that follow
// (softmax, top-k, gate weights) are in route_select.cu.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int TT = ROUTER_TOKENS;     // 64 tokens per block
constexpr int KC = ROUTER_KC;         // 32 hidden columns per stage
constexpr int XS = KC + 4;            // smem row stride of the x tile (floats)

// 256 threads = 16 token groups (4 tokens each) x 16 expert groups; expert group g
// owns experts g, g+16, ..., g+16*(NJ-1).
template <typename TIn, int NJ>
__global__ void __launch_bounds__(256)
router_logits_kernel(const TIn* __restrict__ x, const TIn* __restrict__ wr,
                     float* __restrict__ part, int T, int H, int N, int chunks_per_split) {
  constexpr int NP = 16 * NJ;
  __shared__ __align__(16) float xs[TT * XS];
  __shared__ __align__(16) float ws[KC * NP];
  const int tid = threadIdx.x;
  const int tg = tid >> 4, eg = tid & 15;
  const int t0 = blockIdx.x * TT;
  const int nchunk = H / KC;
  const int c_begin = blockIdx.y * chunks_per_split;
  const int c_end = min(nchunk, c_begin + chunks_per_split);
  pdl_wait();
  pdl_trigger();

  float acc[4][NJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < NJ; ++j) acc[i][j] = 0.f;

  for (int c = c_begin; c < c_end; ++c) {
    const int k0 = c * KC;
    {  // x tile: 64 tokens x 32 columns, 8 elements per thread
      const int t = tid >> 2, kk = (tid & 3) * 8;
      float v[8];
      if (t0 + t < T) {
        load8(x + (size_t)(t0 + t) * H + k0 + kk, v);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
      }
      float* dst = xs + t * XS + kk;
      *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
    for (int i = tid; i < KC * NP; i += 256) {  // W_r columns k0..k0+31 of every expert
      const int e = i / KC, kk = i - e * KC;
      ws[kk * NP + e] = (e < N) ? to_f32(wr[(size_t)e * H + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < KC; kk += 4) {
      float4 xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        xv[i] = *reinterpret_cast<const float4*>(xs + (tg * 4 + i) * XS + kk);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const float w = ws[(kk + q) * NP + eg + 16 * j];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float xq = q == 0 ? xv[i].x : q == 1 ? xv[i].y : q == 2 ? xv[i].z : xv[i].w;
            acc[i][j] = fmaf(xq, w, acc[i][j]);
          }
        }
      }
    }
    __syncthreads();
  }
  float* out = part + (size_t)blockIdx.y * T * N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + tg * 4 + i;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = eg + 16 * j;
      if (t < T && e < N) out[(size_t)t * N + e] = acc[i][j];
    }
  }
}

template <typename TIn>
cudaError_t launch_logits_t(const TIn* x, const TIn* wr, float* part, int T, int H, int N,
                            int ksplit, int cps, cudaStream_t stream) {
  const dim3 grid((T + TT - 1) / TT, ksplit);
  if (N <= 16)
    router_logits_kernel<TIn, 1><<<grid, 256, 0, stream>>>(x, wr, part, T, H, N, cps);
  else if (N <= 32)
    router_logits_kernel<TIn, 2><<<grid, 256, 0, stream>>>(x, wr, part, T, H, N, cps);
  else if (N <= 64)
    router_logits_kernel<TIn, 4><<<grid, 256, 0, stream>>>(x, wr, part, T, H, N, cps);
  else if (N <= 128)
    router_logits_kernel<TIn, 8><<<grid, 256, 0, stream>>>(x, wr, part, T, H, N, cps);
  else
    router_logits_kernel<TIn, 16><<<grid, 256, 0, stream>>>(x, wr, part, T, H, N, cps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits(int dtype, const void* x, const void* w_router, float* part,
                                 int T, int H, int N, int ksplit, int chunks_per_split,
                                 cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (dtype == 1)
    return launch_logits_t(static_cast<const __nv_bfloat16*>(x),
                           static_cast<const __nv_bfloat16*>(w_router), part, T, H, N, ksplit,
                           chunks_per_split, stream);
  return launch_logits_t(static_cast<const float*>(x), static_cast<const float*>(w_router), part,
                         T, H, N, ksplit, chunks_per_split, stream);
}

}  // namespace moe
