// Gate-weighted combine: out[t] = sum over kept slots s of w[t,s] * ye[row(t,s)]
// (cf-1.com/news/5914943 section 2.1 sums the k experts' outputs weighted by the
// gates; devpress.csdn.net MoE page section 4.1 gathers the expert results back into
// token order). Dropped slots contribute nothing and the kept slots keep their weights;
// the residual is added by the caller (cf-1.com/news/5914943 section 2.3 note).
//
// Shared experts (hotelren.com/news/5904824 section 3.3) are slots k..k+S-1 with
// weight 1; a padding token has no row in any slot and gets 0.
//
// One warp per token, 16-byte vectors. The loads of two slots' rows are in flight
// together, held as loaded until they are added; accumulation is fp32 in a fixed slot
// order, so the result does not depend on scheduling.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// MINB: blocks per SM the registers are capped for. 3 (at most 85 registers) keeps 24
// warps' loads in flight per SM on the large layers; a small batch of a few blocks runs
// faster uncapped.
template <typename TIo, int MINB>
__global__ void __launch_bounds__(256, MINB)
combine_kernel(const TIo* __restrict__ ye, const int32_t* __restrict__ slot_row,
               const float* __restrict__ w, int T, int k, int S, int H,
               TIo* __restrict__ out) {
  constexpr int MAX_SLOTS = 32 + MAX_SHARED;
  __shared__ int32_t rows[8][MAX_SLOTS];
  __shared__ float wts[8][MAX_SLOTS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  const int slots = k + S;
  // slot_row and w come from dispatch and the routing kernels, which had completed
  // before the second expert GEMM let this kernel start (that GEMM triggers only after
  // its own wait on the first, which waited on dispatch): read before the wait
  if (t < T)
    for (int sl = lane; sl < slots; sl += 32) {
      rows[warp][sl] = slot_row[(size_t)t * slots + sl];
      wts[warp][sl] = sl < k ? w[(size_t)t * k + sl] : 1.f;
    }
  pdl_wait();  // ye comes from the second expert GEMM
  pdl_trigger();
  if (t >= T) return;
  __syncwarp();
  // Groups of 8 elements (one 16-byte bf16 vector); each lane keeps VPL groups of two
  // slots in flight at once, held as loaded until they are added in slot order.
  constexpr int VPL = 4, SG = 2;
  constexpr int N16 = (int)sizeof(TIo) * 8 / 16;
  const int ngrp = H / 8;
  for (int g0 = 0; g0 < ngrp; g0 += 32 * VPL) {
    float acc[VPL][8];
#pragma unroll
    for (int u = 0; u < VPL; ++u)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
    for (int s0 = 0; s0 < slots; s0 += SG) {
      uint4 raw[SG][VPL][N16];
#pragma unroll
      for (int j = 0; j < SG; ++j) {
        const int r = s0 + j < slots ? rows[warp][s0 + j] : -1;
        if (r < 0) continue;
        const TIo* src = ye + (size_t)r * H;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
          const int g = g0 + u * 32 + lane;
          if (g < ngrp) {
            const uint4* v = reinterpret_cast<const uint4*>(src + g * 8);
#pragma unroll
            for (int i = 0; i < N16; ++i) raw[j][u][i] = v[i];
          }
        }
      }
#pragma unroll
      for (int j = 0; j < SG; ++j) {
        const int r = s0 + j < slots ? rows[warp][s0 + j] : -1;
        if (r < 0) continue;
        const float ws = wts[warp][s0 + j];
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
          const int g = g0 + u * 32 + lane;
          if (g < ngrp) {
            if constexpr (sizeof(TIo) == 2) {
              const uint4 x = raw[j][u][0];
              const uint32_t v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                acc[u][2 * q] = fmaf(ws, bf16_lo(v[q]), acc[u][2 * q]);
                acc[u][2 * q + 1] = fmaf(ws, bf16_hi(v[q]), acc[u][2 * q + 1]);
              }
            } else {
              const uint4 x = raw[j][u][0], y = raw[j][u][N16 - 1];
              const uint32_t v[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[u][q] = fmaf(ws, __uint_as_float(v[q]), acc[u][q]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      const int g = g0 + u * 32 + lane;
      if (g < ngrp) store8(out + (size_t)t * H + g * 8, acc[u]);
    }
  }
}

constexpr int COMBINE_CAPPED_MIN_TOKENS = 4096;

}  // namespace

cudaError_t launch_combine(int dtype, const void* ye, const int32_t* slot_row, const float* w,
                           int T, int k, int S, int H, void* out, cudaStream_t stream,
                           bool pdl) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((T + 7) / 8), block(256);
  // Same-call A/B: capped registers took the Mixtral-shaped combine 48.4 -> 44.5 us and
  // the fine-grained one 36.3 -> 31.5 us, left T = 4096 unchanged and slowed the
  // 64-token decode batch 10.8 -> 12.2 us (its 8 blocks gain nothing from occupancy).
  if (dtype == 1)
    return T >= COMBINE_CAPPED_MIN_TOKENS
               ? launch_kernel(combine_kernel<__nv_bfloat16, 3>, grid, block, 0, stream, pdl,
                               static_cast<const __nv_bfloat16*>(ye), slot_row, w, T, k, S, H,
                               static_cast<__nv_bfloat16*>(out))
               : launch_kernel(combine_kernel<__nv_bfloat16, 1>, grid, block, 0, stream, pdl,
                               static_cast<const __nv_bfloat16*>(ye), slot_row, w, T, k, S, H,
                               static_cast<__nv_bfloat16*>(out));
  return launch_kernel(combine_kernel<float, 1>, grid, block, 0, stream, pdl,
                       static_cast<const float*>(ye), slot_row, w, T, k, S, H,
                       static_cast<float*>(out));
}

}  // namespace moe
