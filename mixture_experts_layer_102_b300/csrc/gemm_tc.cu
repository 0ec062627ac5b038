// bf16 grouped expert GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// The pages batch the experts' matmuls into one grouped call (cf-1.com/news/5914943
// section 3.3, grouped GEMM) and fuse all experts into one kernel that branches on
// the expert id (2kiu.com/news/2885792 section 3.3). Here one persistent launch walks
// a static schedule of (expert row tile, column tile) work items:
//
//   GEMM1 (swiglu): h[r, n0:n0+128] = silu(xp_r W1_e[n0:n0+128]^T) * (xp_r W3_e[n0:n0+128]^T)
//   GEMM1 (gelu):   h[r, n0:n0+256] = gelu(xp_r W1_e[n0:n0+256]^T)
//                   (the two-layer GELU expert, devpress.csdn.net MoE page section 4.1)
//   GEMM2 (plain):  ye[r, n0:n0+256] = h_r W2_e[n0:n0+256]^T
//
// Two tile shapes, one template (CG = CTAs per tile):
//   CG = 1  one CTA per 128-row tile: tcgen05.mma.cta_group::1, M=128 N=256 K=16;
//           per stage the CTA stages 128 A rows and a 256-row B tile made of two
//           128-row boxes (W1 rows n0.. and the matching W3 rows for GEMM1, so gate
//           and up land side by side in every accumulator row; W1 or W2 rows n0..
//           and n0+128.. otherwise): 4 stages of 48 KB.
//   CG = 2  a cluster of two CTAs per 256-row tile: tcgen05.mma.cta_group::2, M=256
//           N=256 K=16; each CTA stages its own 128 A rows and one 128-row half of B
//           (the W1 box in the first CTA, the W3 box in the second), both CTAs' loads
//           complete on the first CTA's full barrier, and the first CTA issues the
//           pair's MMAs and commits them to both CTAs' barriers: 7 stages of 32 KB,
//           a third less shared-memory traffic per SM for the same MMA work.
// Small expert groups favour CG = 1 (less row padding, more tiles to spread over the
// SMs); large ones favour CG = 2.
//
// Per CTA (320 threads):
//   warp 0      TMA producer (128-byte swizzled boxes into the stage ring).
//   warp 1      TMEM allocator; one thread (of the first CTA) issues the MMAs into one
//               of two 256-column fp32 accumulators, so the epilogue of one tile
//               overlaps the main loop of the next (all 512 TMEM columns).
//   warps 2-9   epilogue: two warps per TMEM lane quarter, each taking half of the
//               columns; tcgen05.ld 32 lanes x 16 columns, SwiGLU in fp32, bf16 stores
//               of the rows that belong to the tile's expert.
// Every mbarrier wait is bounded by %globaltimer; a wait that gives up sets the status
// word and an abort flag, the roles drain what they issued, TMEM is freed and the
// kernel returns.
#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BK = 64;                                // 64 bf16 = one 128-byte swizzle row
constexpr int BN = 256;                               // MMA N
constexpr uint32_t BOX_BYTES = 128 * BK * 2;          // one 128-row x 64 box: 16 KB
constexpr int ACC_COLS = 256;
constexpr int NUM_ACC = 2;
constexpr uint32_t TMEM_COLS = 512;
constexpr int GROUP_MAX = 16;                         // most row tiles per raster band
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;

// Shared memory of one CTA, all of it dynamic (the kernel declares no static shared
// memory): from a 1024-byte-aligned base, the stages, then 256 bytes of barriers, the
// TMEM address and the abort flag, then the expert layout tables (first row tile and
// first row of every expert). The allocation adds an allowance for aligning the base;
// the first KB of a CTA's shared memory is reserved, so the dynamic part normally
// starts aligned and the allowance goes unused (the kernel checks it).
constexpr size_t SMEM_OPTIN_MAX = 232448;                     // per-block opt-in limit
template <int CG>
struct Shape {
  static constexpr int TILE_M = 128 * CG;                        // rows per work item
  static constexpr int B_BOXES = 3 - CG;                         // B boxes per CTA stage
  static constexpr uint32_t STAGE_BYTES = BOX_BYTES * (1 + B_BOXES);  // 48 KB or 32 KB
  static constexpr int STAGES = CG == 1 ? 4 : 7;
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 2 * NUM_ACC + 1) + 8;
  static_assert(BAR_BYTES <= 256, "barrier area");
  static constexpr size_t TABLE_OFFSET = (size_t)STAGES * STAGE_BYTES + 256;
  static constexpr size_t CARVE_BYTES = TABLE_OFFSET + 2 * (MAX_EXPERTS + 1) * 4;
  static constexpr size_t PAD_BYTES =
      SMEM_OPTIN_MAX - CARVE_BYTES < 1024 ? SMEM_OPTIN_MAX - CARVE_BYTES : 1024;
  static constexpr size_t SMEM_BYTES = CARVE_BYTES + PAD_BYTES;
  static_assert(CARVE_BYTES <= SMEM_OPTIN_MAX, "shared memory");
};

// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9 = 1),
// B bf16 (bits 10-12 = 1), A and B K-major (bits 15, 16 = 0), N>>3 at bits 17-22,
// M>>4 at bits 24-28 (M = 128 per CTA, or 256 for a CTA pair).
template <int CG>
__host__ __device__ constexpr uint32_t idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)((128 * CG) >> 4) << 24);
}

// silu(z) = z / (1 + e^-z) with the fast intrinsics: their error (a few ulp of fp32)
// is far below the bf16 rounding of h that follows. e^-z overflows to +inf for very
// negative z and the quotient then reads 0, the limit of silu.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Exact GELU, z * Phi(z) = z/2 * (1 + erf(z / sqrt 2)).
__device__ __forceinline__ float gelu_erf(float z) {
  return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}

// Work item w -> (expert, row tile, column tile). Items are grouped by expert (an
// expert's tiles x all column tiles, experts in order); inside an expert, bands of
// row tiles sweep the column tiles with the row tile fastest, so the units in flight
// share a few A tiles and each weight tile of the expert is streamed about once per
// band. An expert of `tiles` row tiles gets ceil(tiles / GROUP_MAX) bands whose
// heights differ by at most one: a lone short band at the end would stream the
// expert's whole weight set once more for a few rows. `tfirst` [N+1] holds each
// expert's first row tile (shared memory).
__device__ __forceinline__ void raster(int w, const int32_t* tfirst, int N, int n_tiles, int& e,
                                       int& mt, int& nt) {
  int lo = 0, hi = N - 1;  // last expert whose first item is <= w
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tfirst[mid] * n_tiles <= w) lo = mid; else hi = mid - 1;
  }
  const int t0 = tfirst[lo];
  const int tiles = tfirst[lo + 1] - t0;  // >= 1: w lies in this expert's items
  const int local = w - t0 * n_tiles;
  const int nb = (tiles + GROUP_MAX - 1) / GROUP_MAX;
  const int base = tiles / nb, rem = tiles - base * nb;  // rem bands of base + 1 rows
  const int r = local / n_tiles;  // the band holding item `local` holds row tile r
  const int band = r < rem * (base + 1) ? r / (base + 1) : rem + (r - rem * (base + 1)) / base;
  const int m_first = band * base + min(band, rem);
  const int gm = base + (band < rem ? 1 : 0);
  const int in_band = local - m_first * n_tiles;
  mt = t0 + m_first + in_band % gm;
  nt = in_band / gm;
  e = lo;
}

struct TcArgs {
  const int32_t* offsets;
  const int32_t* num_mtiles;
  const int32_t* tile_first;  // [N+1] first row tile of each expert
  int N;
  __nv_bfloat16* out;
  int out_ld;        // output row stride (elements)
  int K;             // reduction length, multiple of 64
  int n_tiles;       // column tiles
  int n_per_tile;    // output columns per tile: 128 (swiglu) or 256
  int n_valid;       // output columns in total
  int b1_row_off;    // row offset of the second CTA's B box: 0 (W3) or 128 (W2)
  uint32_t* status;
#ifdef MOE_TEST_HOOKS
  int test_skip_kchunk;  // k-chunk of CTA 0's first item whose loads are withheld, -1: none
#endif
};

template <int EPI, int CG>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, TcArgs a) {
  using S = Shape<CG>;
  extern __shared__ uint8_t smem_raw[];
  // Every CTA carves the same offsets (same dynamic size and alignment rule), which
  // the pair MMA relies on: its descriptors address both CTAs' tiles at once.
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  if (base - raw > S::PAD_BYTES) {  // the carve would pass the allocation: refuse
    if (threadIdx.x == 0) report(a.status, STATUS_BAD_LAYOUT);
    return;
  }
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t full_bar = base + S::STAGES * S::STAGE_BYTES;  // [STAGES] (first CTA's used)
  const uint32_t empty_bar = full_bar + 8 * S::STAGES;           // [STAGES]
  const uint32_t accf_bar = empty_bar + 8 * S::STAGES;           // [NUM_ACC]
  const uint32_t acce_bar = accf_bar + 8 * NUM_ACC;              // [NUM_ACC] (first CTA's used)
  const uint32_t drain_bar = acce_bar + 8 * NUM_ACC;             // [1]
  int* misc = reinterpret_cast<int*>(base_ptr + S::STAGES * S::STAGE_BYTES +
                                     8 * (2 * S::STAGES + 2 * NUM_ACC + 1));
  // misc[0]: TMEM base address, misc[1]: abort flag
  volatile int* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(full_bar + 8 * s, 1);
      mbar_init(empty_bar + 8 * s, 1);
    }
    for (int i = 0; i < NUM_ACC; ++i) {
      mbar_init(accf_bar + 8 * i, 1);
      mbar_init(acce_bar + 8 * i, EPI_WARPS * CG);  // one arrive per epilogue warp
    }
    mbar_init(drain_bar, 1);
    misc[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&tmA);
    prefetch_map(&tmB0);
    prefetch_map(&tmB1);
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(misc)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(misc)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  // The expert layout comes from the routing kernels, which ran two or more launches
  // before this one and have completed; only the A rows (the previous kernel's output)
  // need the wait below.
  int32_t* tfirst = reinterpret_cast<int32_t*>(base_ptr + S::TABLE_OFFSET);  // [N+1]
  int32_t* roff = tfirst + (MAX_EXPERTS + 1);                                  // [N+1]
  for (int i = threadIdx.x; i <= a.N; i += blockDim.x) {
    tfirst[i] = a.tile_first[i];
    roff[i] = a.offsets[i];
  }
  tc_fence_before();
  if constexpr (CG == 2) cluster_sync();  // both CTAs' barriers, TMEM and tables ready
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = static_cast<uint32_t>(misc[0]);
  const int num_mt = *a.num_mtiles;
  if (threadIdx.x != 0) {  // the producer (thread 0) waits after its first weight loads
    pdl_wait();
    pdl_trigger();
  }
  const int total = num_mt * a.n_tiles;
  const int kchunks = a.K / BK;
  const int unit = blockIdx.x / CG;       // CTA (CG = 1) or CTA pair (CG = 2)
  const int num_units = gridDim.x / CG;

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------- TMA producer
      // CG = 2: both CTAs' loads complete on the first CTA's full barriers.
      const uint32_t full_c = CG == 2 ? map_to_cta(full_bar, 0) : full_bar;
      // Weight boxes of k-chunk kc of expert e, column tile n0, into stage sA.
      auto load_b = [&](uint32_t sA, uint32_t fb, int kc, int n0, int e) {
        if constexpr (CG == 2) {
          if (leader) tma_load_3d<CG>(sA + BOX_BYTES, &tmB0, fb, kc * BK, n0, e);
          else tma_load_3d<CG>(sA + BOX_BYTES, &tmB1, fb, kc * BK, n0 + a.b1_row_off, e);
        } else {
          tma_load_3d<CG>(sA + BOX_BYTES, &tmB0, fb, kc * BK, n0, e);
          tma_load_3d<CG>(sA + 2 * BOX_BYTES, &tmB1, fb, kc * BK, n0 + a.b1_row_off, e);
        }
      };
      // The weights are the caller's: the first unit's weight boxes for the first
      // STAGES k-chunks go out before the wait for the previous kernel (the stages are
      // fresh, so no empty-barrier wait is due), and only their A boxes follow it.
#ifdef MOE_TEST_HOOKS
      // Test builds only: on single-CTA tiles, CTA 0 issues no load (and no expected
      // byte count) for one k-chunk of its first work item. That stage's full barrier
      // then never completes, the MMA thread's bounded wait gives up, and the abort
      // path runs: nothing is in flight for the withheld stage.
      const int skip_kc = (CG == 1 && blockIdx.x == 0) ? a.test_skip_kchunk : -1;
#else
      constexpr int skip_kc = -1;
#endif
      int pre = 0;
      if (unit < total) {
        int e, mt, nt;
        raster(unit, tfirst, a.N, a.n_tiles, e, mt, nt);
        pre = min(S::STAGES, kchunks);
        for (int kc = 0; kc < pre; ++kc) {
          if (kc == skip_kc) continue;
          if (leader) mbar_expect_tx(full_bar + 8 * kc, CG * S::STAGE_BYTES);
          load_b(base + kc * S::STAGE_BYTES, full_c + 8 * kc, kc, nt * a.n_per_tile, e);
        }
      }
      pdl_wait();
      pdl_trigger();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_parity = 0;
      bool ok = true;
      for (int w = unit; w < total && ok; w += num_units) {
        int e, mt, nt;
        raster(w, tfirst, a.N, a.n_tiles, e, mt, nt);
        const int row0 = roff[e] + (mt - tfirst[e]) * S::TILE_M + (int)rank * 128;
        const int n0 = nt * a.n_per_tile;
        for (int kc = 0; kc < kchunks; ++kc, ++issued) {
          const uint32_t sA = base + stage * S::STAGE_BYTES;
          const uint32_t fb = full_c + 8 * stage;
          if (!(w == unit && kc == skip_kc)) {
            if (issued >= pre) {
              if (!mbar_wait(empty_bar + 8 * stage, phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                ok = false;
                break;
              }
              if (leader) mbar_expect_tx(full_bar + 8 * stage, CG * S::STAGE_BYTES);
              load_b(sA, fb, kc, n0, e);
            }
            tma_load_2d<CG>(sA, &tmA, fb, kc * BK, row0);
            used |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == S::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        report(a.status, STATUS_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      // Let every load this CTA issued land before the CTA may exit: the first CTA's
      // full barriers count all bytes; the second CTA sees a stage consumed (hence
      // landed) when the MMA's commit frees it.
      for (int s = 0; s < S::STAGES; ++s) {
        if (!((used >> s) & 1u)) continue;
        const uint32_t par = (last_parity >> s) & 1u;
        if (leader) mbar_wait(full_bar + 8 * s, par, nullptr, DRAIN_LIMIT_NS);
        else mbar_wait(empty_bar + 8 * s, par, nullptr, DRAIN_LIMIT_NS);
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {  // ------------------------------------ MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int w = unit; w < total && ok; w += num_units) {
        if (!mbar_wait(acce_bar + 8 * acc, acc_phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * ACC_COLS);
        for (int kc = 0; kc < kchunks; ++kc) {
          if (!mbar_wait(full_bar + 8 * stage, phase, abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = base + stage * S::STAGE_BYTES;
          const uint64_t da = sw128_desc(sA);
          const uint64_t db = sw128_desc(sA + BOX_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes of K per step
            tc_mma<CG>(d, da + 2 * kk, db + 2 * kk, idesc<CG>(), (kc | kk) != 0 ? 1u : 0u);
          tc_commit<CG>(empty_bar + 8 * stage);
          if (++stage == S::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit<CG>(accf_bar + 8 * acc);
        if (++acc == NUM_ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        report(a.status, STATUS_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      // Every MMA issued above has completed once this barrier flips.
      tc_commit_own<CG>(drain_bar);
      mbar_wait(drain_bar, 0, nullptr, DRAIN_LIMIT_NS);
    }
  } else {  // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;        // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;    // which half of the columns
    const int row_in_cta = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t acce_c = CG == 2 ? map_to_cta(acce_bar, 0) : acce_bar;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = unit; w < total; w += num_units) {
      int e, mt, nt;
      raster(w, tfirst, a.N, a.n_tiles, e, mt, nt);
      const int r = roff[e] + (mt - tfirst[e]) * S::TILE_M + (int)rank * 128 + row_in_cta;
      const bool valid = r < roff[e + 1];
      bool ok = mbar_wait(accf_bar + 8 * acc, acc_phase, abort_flag, WAIT_LIMIT_NS);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          report(a.status, STATUS_WAIT_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t t = tmem_base + lane_addr + (uint32_t)(acc * ACC_COLS);
      __nv_bfloat16* orow = a.out + (size_t)r * a.out_ld + (size_t)nt * a.n_per_tile;
      const int cols_left = a.n_valid - nt * a.n_per_tile;
      if constexpr (EPI == EPI_SWIGLU) {  // h columns [64*half, 64*half + 64): gate at c, up at 128 + c
#pragma unroll 1
        for (int c = 64 * half; c < 64 * half + 64; c += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(t + c, g);
          tmem_ld16(t + 128 + c, u);
          tmem_wait_ld();
          if (valid && c < cols_left) {
            uint32_t p[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float h0 = silu_fast(__uint_as_float(g[2 * q])) * __uint_as_float(u[2 * q]);
              const float h1 =
                  silu_fast(__uint_as_float(g[2 * q + 1])) * __uint_as_float(u[2 * q + 1]);
              p[q] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
            dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
          }
        }
      } else {  // columns [128*half, 128*half + 128) of ye (plain) or h (gelu)
#pragma unroll 1
        for (int c = 128 * half; c < 128 * half + 128; c += 16) {
          uint32_t v[16];
          tmem_ld16(t + c, v);
          tmem_wait_ld();
          if (valid && c < cols_left) {
            uint32_t p[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float v0 = __uint_as_float(v[2 * q]), v1 = __uint_as_float(v[2 * q + 1]);
              if constexpr (EPI == EPI_GELU) {
                v0 = gelu_erf(v0);
                v1 = gelu_erf(v1);
              }
              p[q] = pack_bf16x2(v0, v1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
            dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) mbar_arrive_cluster(acce_c + 8 * acc);
        else mbar_arrive(acce_c + 8 * acc);
      }
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // no CTA leaves while its peer may signal it
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(TMEM_COLS)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(TMEM_COLS)
                   : "memory");
  }
}

// ------------------------------------------------------------------ host side

#ifdef MOE_TEST_HOOKS
int g_test_skip_kchunk = -1;  // see moe_test_withhold_gemm_load
#endif

// Work units (CTAs, or CTA pairs) that can be resident at once: the grid size.
template <int EPI, int CG>
int grid_units() {
  static std::atomic<int> cached[64];  // 0 until the first launch on that device
  int dev = 0;
  cudaGetDevice(&dev);
  const int c = dev >= 0 && dev < 64 ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (c > 0) return c;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int n = sms > 0 ? sms / CG : 1;
  if (CG == 2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Shape<CG>::SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, grouped_gemm_tc_kernel<EPI, CG>, &cfg) ==
            cudaSuccess &&
        c > 0)
      n = c;
    cudaGetLastError();
  }
  if (n < 1) n = 1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int EPI, int CG>
cudaError_t launch_t(const CUtensorMap& mA, const CUtensorMap& mB0, const CUtensorMap& mB1,
                     const TcArgs& t, cudaStream_t stream, bool pdl) {
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(grouped_gemm_tc_kernel<EPI, CG>),
                                      Shape<CG>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CG * grid_units<EPI, CG>(), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Shape<CG>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (CG == 2) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = CG;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  e = cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<EPI, CG>, mA, mB0, mB1, t);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_tc(const GroupedGemmArgs& a, cudaStream_t stream, bool pdl) {
  if (a.max_mtiles == 0 || a.A_rows == 0) return cudaSuccess;
  if (a.N > MAX_EXPERTS) return cudaErrorInvalidValue;
  const bool swiglu = a.epi == EPI_SWIGLU;
  CUtensorMap mA, mB0, mB1;
  if (!make_map(&mA, a.A, 2, (uint64_t)a.K, 0, (uint64_t)a.A_rows)) return cudaErrorInvalidValue;
  if (!make_map(&mB0, a.B0, 3, (uint64_t)a.K, (uint64_t)a.n_cols, (uint64_t)a.N))
    return cudaErrorInvalidValue;
  if (!make_map(&mB1, swiglu ? a.B1 : a.B0, 3, (uint64_t)a.K, (uint64_t)a.n_cols, (uint64_t)a.N))
    return cudaErrorInvalidValue;
  TcArgs t;
  t.offsets = a.offsets;
  t.num_mtiles = a.num_mtiles;
  t.tile_first = a.tile_first;
  t.N = a.N;
  t.out = static_cast<__nv_bfloat16*>(a.out);
  t.out_ld = a.n_cols;
  t.K = a.K;
  t.n_per_tile = swiglu ? 128 : 256;
  t.n_tiles = (a.n_cols + t.n_per_tile - 1) / t.n_per_tile;
  t.n_valid = a.n_cols;
  t.b1_row_off = swiglu ? 0 : 128;
  t.status = a.status;
#ifdef MOE_TEST_HOOKS
  t.test_skip_kchunk = g_test_skip_kchunk;
#endif
  switch (a.epi) {
    case EPI_SWIGLU:
      return a.pair ? launch_t<EPI_SWIGLU, 2>(mA, mB0, mB1, t, stream, pdl)
                    : launch_t<EPI_SWIGLU, 1>(mA, mB0, mB1, t, stream, pdl);
    case EPI_GELU:
      return a.pair ? launch_t<EPI_GELU, 2>(mA, mB0, mB1, t, stream, pdl)
                    : launch_t<EPI_GELU, 1>(mA, mB0, mB1, t, stream, pdl);
    default:
      return a.pair ? launch_t<EPI_PLAIN, 2>(mA, mB0, mB1, t, stream, pdl)
                    : launch_t<EPI_PLAIN, 1>(mA, mB0, mB1, t, stream, pdl);
  }
}

}  // namespace moe

#ifdef MOE_TEST_HOOKS
extern "C" void moe_test_withhold_gemm_load(int kchunk) { moe::g_test_skip_kchunk = kchunk; }
#endif
