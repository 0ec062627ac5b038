// float32 grouped expert GEMM on CUDA cores, used when the layer's dtype is float32:
// fp32 FMA throughout (no TF32), so the result stays within fp32 rounding of the
// exact product. Expert e's rows are [offsets[e], offsets[e+1]) of the permuted
// buffer, visited as 128-row tiles from the tile table the capacity scan writes.
//
//   swiglu: out = silu(A W1_e^T) * (A W3_e^T)   (2kiu.com/news/2885792 section 2.2)
//   gelu:   out = gelu(A W1_e^T), exact erf GELU (devpress.csdn.net MoE page section 4.1)
//   plain:  out = A W2_e^T
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = TILE_ROWS_1;  // 128 rows: one tile of the 128-row table per block
constexpr int BN = 64;           // output columns per block
constexpr int BK = 16;

template <int EPI>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ B0,
                 const float* __restrict__ B1, float* __restrict__ out, int K, int n_cols,
                 int N, const int32_t* __restrict__ tile_first,
                 const int32_t* __restrict__ offsets, const int32_t* __restrict__ num_mtiles) {
  constexpr bool SWIGLU = EPI == EPI_SWIGLU;
  const int mt = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  if (mt >= *num_mtiles) return;
  __shared__ int32_t tfirst[MAX_EXPERTS + 1];
  for (int i = threadIdx.x; i <= N; i += blockDim.x) tfirst[i] = tile_first[i];
  __syncthreads();
  int e = 0, hi = N - 1;  // the expert of row tile mt: last e with tfirst[e] <= mt
  while (e < hi) {
    const int mid = (e + hi + 1) >> 1;
    if (tfirst[mid] <= mt) e = mid; else hi = mid - 1;
  }
  const int r0 = offsets[e] + (mt - tfirst[e]) * BM;
  const int rend = offsets[e + 1];
  const int n0 = blockIdx.y * BN;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs0[BK][BN + 4];
  __shared__ float Bs1[SWIGLU ? BK : 1][BN + 4];
  const float* Be0 = B0 + (size_t)e * n_cols * K;
  const float* Be1 = SWIGLU ? B1 + (size_t)e * n_cols * K : nullptr;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;  // rows ty*8.., cols tx*4..
  float acc0[8][4], acc1[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc0[i][j] = acc1[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int l = tid; l < BM * BK; l += 256) {
      const int r = l / BK, kk = l - r * BK;
      As[kk][r] = (r0 + r < rend) ? A[(size_t)(r0 + r) * K + k0 + kk] : 0.f;
    }
    for (int l = tid; l < BN * BK; l += 256) {
      const int n = l / BK, kk = l - n * BK;
      const bool ok = n0 + n < n_cols;
      Bs0[kk][n] = ok ? Be0[(size_t)(n0 + n) * K + k0 + kk] : 0.f;
      if (SWIGLU) Bs1[kk][n] = ok ? Be1[(size_t)(n0 + n) * K + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[8], b0[4], b1[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) av[i] = As[kk][ty * 8 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b0[j] = Bs0[kk][tx * 4 + j];
        b1[j] = SWIGLU ? Bs1[kk][tx * 4 + j] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = fmaf(av[i], b0[j], acc0[i][j]);
          if (SWIGLU) acc1[i][j] = fmaf(av[i], b1[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + ty * 8 + i;
    if (r >= rend) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx * 4 + j;
      if (c >= n_cols) continue;
      float v = acc0[i][j];
      if constexpr (EPI == EPI_SWIGLU) v = silu(v) * acc1[i][j];
      if constexpr (EPI == EPI_GELU) v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
      out[(size_t)r * n_cols + c] = v;
    }
  }
}

}  // namespace

cudaError_t launch_grouped_gemm_simt(const GroupedGemmArgs& a, cudaStream_t stream) {
  if (a.max_mtiles == 0) return cudaSuccess;
  const dim3 grid(a.max_mtiles, (a.n_cols + BN - 1) / BN);
  const float* A = static_cast<const float*>(a.A);
  const float* B0 = static_cast<const float*>(a.B0);
  float* out = static_cast<float*>(a.out);
  if (a.epi == EPI_SWIGLU)
    gemm_simt_kernel<EPI_SWIGLU><<<grid, 256, 0, stream>>>(
        A, B0, static_cast<const float*>(a.B1), out, a.K, a.n_cols, a.N, a.tile_first,
        a.offsets, a.num_mtiles);
  else if (a.epi == EPI_GELU)
    gemm_simt_kernel<EPI_GELU><<<grid, 256, 0, stream>>>(A, B0, nullptr, out, a.K, a.n_cols,
                                                         a.N, a.tile_first, a.offsets,
                                                         a.num_mtiles);
  else
    gemm_simt_kernel<EPI_PLAIN><<<grid, 256, 0, stream>>>(A, B0, nullptr, out, a.K, a.n_cols,
                                                          a.N, a.tile_first, a.offsets,
                                                          a.num_mtiles);
  return cudaGetLastError();
}

}  // namespace moe
