// bf16 router logits on the sm_103a tensor cores: logits = x W_r^T, the small linear
// layer of the router (cf-1.com/news/5914943 section 2.1; 2kiu.com/news/2885792
// section 3.1), as split-K fp32 partials part[split][t][e]. W_r is [N, H], the
// nn.Linear [out, in] orientation, so both MMA operands are K-major 128-byte-swizzled
// TMA tiles read straight from the caller's tensors.
//
// The product is thin (N <= 256 columns against H-long rows of x), so it is bound by
// reading x once from HBM; on CUDA cores the fine-grained layer's 64 experts made it
// compute-bound instead. One CTA per (128-token tile, K slice): warp 0 streams x and
// W_r boxes through a 4-stage TMA ring (the W_r box is N_pad = N rounded up to 16 rows;
// TMA fills the rows past N with zeros), one thread of warp 1 issues
// tcgen05.mma.cta_group::1 (M=128, N=N_pad, K=16) into a TMEM accumulator, warps 2-5
// read it back (one token per thread) and store the fp32 partial logits of the real
// experts. The K slices fill the GPU when T is small (decode); the routing-decision
// kernel sums the slices in a fixed order. Waits are bounded as in the expert GEMM.
#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BK = 64;                           // 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = 128 * BK * 2;       // 16 KB: 128 tokens x 64
constexpr int NUM_THREADS = 192;

struct RouterTcArgs {
  float* part;
  int T, N, n_pad;
  int kc_per_split, kc_total;
  uint32_t idesc;
  uint32_t tmem_cols;
  uint32_t b_bytes;       // one W_r box: n_pad rows x 128 bytes
  uint32_t stage_bytes;   // A box + B box, rounded up to 1024
  uint32_t* status;
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 RouterTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t full_bar = base + STAGES * a.stage_bytes;
  const uint32_t empty_bar = full_bar + 8 * STAGES;
  const uint32_t accf_bar = empty_bar + 8 * STAGES;
  int* misc = reinterpret_cast<int*>(base_ptr + STAGES * a.stage_bytes + 8 * (2 * STAGES + 1));
  volatile int* abort_flag = misc + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128;
  const int split = blockIdx.y;
  const int kc0 = split * a.kc_per_split;
  const int kc1 = min(a.kc_total, kc0 + a.kc_per_split);

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
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
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
      for (int kc = kc0; kc < kc1; ++kc) {
        if (!mbar_wait(empty_bar + 8 * stage, phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const uint32_t sA = base + stage * a.stage_bytes;
        const uint32_t fb = full_bar + 8 * stage;
        mbar_expect_tx(fb, A_BYTES + a.b_bytes);
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
        report(a.status, STATUS_WAIT_TIMEOUT);
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
      for (int kc = kc0; kc < kc1; ++kc) {
        if (!mbar_wait(full_bar + 8 * stage, phase, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sA = base + stage * a.stage_bytes;
        const uint64_t da = sw128_desc(sA);
        const uint64_t db = sw128_desc(sA + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma<1>(tmem, da + 2 * kk, db + 2 * kk, a.idesc, (kc > kc0 || kk > 0) ? 1u : 0u);
        tc_commit<1>(empty_bar + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        report(a.status, STATUS_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      tc_commit<1>(accf_bar);  // also drains: every MMA above is complete when it flips
    }
  } else {  // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int t = m0 + quarter * 32 + lane;
    bool ok = mbar_wait(accf_bar, 0, abort_flag, WAIT_LIMIT_NS);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
      float* row = a.part + ((size_t)split * a.T + t) * a.N;
      for (int c = 0; c < a.n_pad; c += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + c, v);
        tmem_wait_ld();
        if (t < a.T) {
#pragma unroll
          for (int q = 0; q < 16; ++q)
            if (c + q < a.N) row[c + q] = __uint_as_float(v[q]);
        }
      }
    } else if (lane == 0) {
      report(a.status, STATUS_WAIT_TIMEOUT);
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(a.tmem_cols)
                 : "memory");
  }
}

}  // namespace

int router_tc_npad(int N) { return (N + 15) / 16 * 16; }

void router_tc_split(int T, int H, int* ksplit, int* kc_per_split) {
  const int mt = (T + 127) / 128;
  const int kc_total = H / BK;
  int ks = mt > 0 ? (148 + mt / 2) / mt : 1;  // about one CTA per SM
  if (ks > 16) ks = 16;
  if (ks > kc_total) ks = kc_total;
  if (ks < 1) ks = 1;
  *kc_per_split = (kc_total + ks - 1) / ks;
  *ksplit = (kc_total + *kc_per_split - 1) / *kc_per_split;
}

cudaError_t launch_router_logits_tc(const void* x, const void* w_router, float* part, int T,
                                    int H, int N, uint32_t* status, cudaStream_t stream,
                                    bool pdl) {
  if (T == 0) return cudaSuccess;
  const int n_pad = router_tc_npad(N);
  CUtensorMap mX, mW;
  if (!make_map(&mX, x, 2, (uint64_t)H, 0, (uint64_t)T, 128)) return cudaErrorInvalidValue;
  if (!make_map(&mW, w_router, 2, (uint64_t)H, 0, (uint64_t)N, (uint32_t)n_pad))
    return cudaErrorInvalidValue;
  RouterTcArgs a;
  a.part = part;
  a.T = T;
  a.N = N;
  a.n_pad = n_pad;
  int ksplit = 1;
  router_tc_split(T, H, &ksplit, &a.kc_per_split);
  a.kc_total = H / BK;
  // kind::f16 descriptor: D fp32, A/B bf16, K-major, N = n_pad, M = 128
  a.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n_pad >> 3) << 17) |
            ((uint32_t)(128 >> 4) << 24);
  uint32_t cols = 32;
  while ((int)cols < n_pad) cols <<= 1;
  a.tmem_cols = cols;
  a.b_bytes = (uint32_t)n_pad * 128;
  a.stage_bytes = (A_BYTES + a.b_bytes + 1023u) & ~1023u;
  a.status = status;
  const size_t smem = 1024 + (size_t)STAGES * a.stage_bytes + 256;
  const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(router_tc_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(router_tc_kernel, dim3((T + 127) / 128, ksplit), dim3(NUM_THREADS), smem,
                       stream, pdl, mX, mW, a);
}

}  // namespace moe
