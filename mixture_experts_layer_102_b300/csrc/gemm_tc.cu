// bf16 grouped expert GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA),
// two SMs per tile.
//
// The pages batch the experts' matmuls into one grouped call (cf-1.com/news/5914943
// section 3.3, grouped GEMM) and fuse all experts into one kernel that branches on
// the expert id (2kiu.com/news/2885792 section 3.3). Here one persistent launch walks
// a static schedule of (expert row tile, column tile) work items:
//
//   GEMM1 (swiglu): h[r, n0:n0+128] = silu(xp_r W1_e[n0:n0+128]^T) * (xp_r W3_e[n0:n0+128]^T)
//   GEMM2 (plain):  ye[r, n0:n0+256] = h_r W2_e[n0:n0+256]^T
//
// A cluster of two CTAs (one per SM) computes one 256-row x 256-column tile with
// tcgen05.mma.cta_group::2 (M=256, N=256, K=16): each CTA stages its own 128 rows of
// A and one 128-row half of B (W1 rows in the first CTA and the matching W3 rows in
// the second for GEMM1, so gate and up land side by side in every accumulator row;
// W2 rows n0.. and n0+128.. for GEMM2), and each CTA's TMEM holds the fp32
// accumulator of its own 128 rows. Per CTA (192 threads):
//   warp 0      TMA producer: 6-stage ring of 32 KB stages (A box + B box, 128-byte
//               swizzle); both CTAs' loads complete on the first CTA's full barrier.
//   warp 1      TMEM allocation (both CTAs); in the first CTA one thread issues the
//               pair's MMAs and commits them to both CTAs' barriers (multicast).
//   warps 2-5   epilogue: tcgen05.ld 32 lanes x 16 columns of its own TMEM, SwiGLU in
//               fp32, bf16 stores of the rows that belong to the tile's expert; then
//               one arrive per warp on the first CTA's accumulator-empty barrier.
// Two 256-column accumulators per CTA (all 512 TMEM columns) let the epilogue of one
// tile overlap the main loop of the next. Every mbarrier wait is bounded by
// %globaltimer; a wait that gives up sets the status word and an abort flag, the
// roles drain what they issued, TMEM is freed and the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = GEMM_BM;                           // 256 rows per tile (128 per CTA)
constexpr int BK = 64;                                // 64 bf16 = one 128-byte swizzle row
constexpr int BN = 256;                               // MMA N (128 B rows per CTA)
constexpr int STAGES = 6;
constexpr uint32_t A_BYTES = 128 * BK * 2;            // 16 KB: this CTA's 128 A rows
constexpr uint32_t B_BYTES = 128 * BK * 2;            // 16 KB: this CTA's half of B
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;   // 32 KB
constexpr int ACC_COLS = 256;
constexpr int NUM_ACC = 2;
constexpr uint32_t TMEM_COLS = 512;
constexpr int GROUP_M = 8;                            // row tiles per raster band
constexpr int NUM_THREADS = 192;
constexpr int BAR_BYTES = 8 * (2 * STAGES + 2 * NUM_ACC + 1) + 16;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;     // 2 s
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;     // 0.2 s
static_assert(BAR_BYTES <= 256, "barrier area");
static_assert(BM == 256, "one tile = two CTAs x 128 TMEM lanes");

// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9 = 1),
// B bf16 (bits 10-12 = 1), A and B K-major (bits 15, 16 = 0), N>>3 at bits 17-22,
// M>>4 at bits 24-28; M = 256 is the pair's M.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                           ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Arrive on a barrier given by its shared::cluster address (this CTA's or the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete. Gives up (returns false)
// after `limit_ns`, or early once another role of this CTA raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int* abort_flag, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// TMA tile loads into this CTA's shared memory, completing on a barrier that may be
// in either CTA of the pair (cta_group::2).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t cbar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cbar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t cbar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cbar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on the barrier at this shared-memory offset in both CTAs of the pair
// when all MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)0x3)
      : "memory");
}
// Arrive once on this CTA's barrier when all MMAs issued so far have completed.
__device__ __forceinline__ void tc_commit_own(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(IDESC), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand stored as 128-byte rows
// (64 bf16 of K) with the 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)   // start address >> 4
         | ((uint64_t)1 << 16)                  // leading byte offset (unused here)
         | ((uint64_t)(1024 >> 4) << 32)        // stride byte offset: 8 rows x 128 B
         | ((uint64_t)1 << 46)                  // tcgen05 descriptor version
         | ((uint64_t)2 << 61);                 // 128-byte swizzle
}

// Work item w -> (row tile, column tile): bands of GROUP_M row tiles, row tile
// fastest inside a band, so the pairs in flight share a few A and B tiles in L2.
__device__ __forceinline__ void raster(int w, int num_mt, int n_tiles, int& mt, int& nt) {
  const int band_size = GROUP_M * n_tiles;
  const int band = w / band_size;
  const int local = w - band * band_size;
  const int m_first = band * GROUP_M;
  const int gm = min(GROUP_M, num_mt - m_first);
  mt = m_first + local % gm;
  nt = local / gm;
}

struct TcArgs {
  const int32_t* tile_expert;
  const int32_t* tile_row0;
  const int32_t* offsets;
  const int32_t* num_mtiles;
  __nv_bfloat16* out;
  int out_ld;        // output row stride (elements)
  int K;             // reduction length, multiple of 64
  int n_tiles;       // column tiles
  int n_per_tile;    // output columns per tile: 128 (swiglu) or 256
  int n_valid;       // output columns in total
  int b1_row_off;    // row offset of the second CTA's B box: 0 (W3) or 128 (W2)
  uint32_t* status;
};

template <bool SWIGLU>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // Both CTAs carve the same offsets (same dynamic size and alignment rule), which
  // the pair MMA relies on: its descriptors address both CTAs' tiles at once.
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t full_bar = base + STAGES * STAGE_BYTES;  // [STAGES] (used in CTA 0)
  const uint32_t empty_bar = full_bar + 8 * STAGES;        // [STAGES]
  const uint32_t accf_bar = empty_bar + 8 * STAGES;        // [NUM_ACC]
  const uint32_t acce_bar = accf_bar + 8 * NUM_ACC;        // [NUM_ACC] (used in CTA 0)
  const uint32_t drain_bar = acce_bar + 8 * NUM_ACC;       // [1]
  int* misc = reinterpret_cast<int*>(base_ptr + STAGES * STAGE_BYTES + 8 * (2 * STAGES + 2 * NUM_ACC + 1));
  // misc[0]: TMEM base address, misc[1]: abort flag
  volatile int* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar + 8 * s, 1);
      mbar_init(empty_bar + 8 * s, 1);
    }
    for (int i = 0; i < NUM_ACC; ++i) {
      mbar_init(accf_bar + 8 * i, 1);
      mbar_init(acce_bar + 8 * i, 8);  // one arrive per epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    misc[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&tmA);
    prefetch_map(&tmB0);
    prefetch_map(&tmB1);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(misc)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = static_cast<uint32_t>(misc[0]);

  const int num_mt = *a.num_mtiles;
  const int total = num_mt * a.n_tiles;
  const int kchunks = a.K / BK;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------- TMA producer
      const uint32_t full_c = map_to_cta(full_bar, 0);  // the leader's full barriers
      const CUtensorMap* mapB = leader ? &tmB0 : &tmB1;
      const int b_off = leader ? 0 : a.b1_row_off;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_parity = 0;
      bool ok = true;
      for (int w = pair; w < total && ok; w += num_pairs) {
        int mt, nt;
        raster(w, num_mt, a.n_tiles, mt, nt);
        const int e = a.tile_expert[mt];
        const int row0 = a.tile_row0[mt] + (int)rank * 128;
        const int n0 = nt * a.n_per_tile + b_off;
        for (int kc = 0; kc < kchunks; ++kc) {
          if (!mbar_wait(empty_bar + 8 * stage, phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          const uint32_t sA = base + stage * STAGE_BYTES;
          const uint32_t fb = full_c + 8 * stage;
          if (leader) mbar_expect_tx(full_bar + 8 * stage, 2 * STAGE_BYTES);
          tma_load_2d(sA, &tmA, fb, kc * BK, row0);
          tma_load_3d(sA + A_BYTES, mapB, fb, kc * BK, n0, e);
          used |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        report(a.status, STATUS_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      // Let every load this CTA issued land before the CTA may exit: the leader's full
      // barriers count both CTAs' bytes; the peer sees a stage consumed (hence landed)
      // when the MMA's commit frees it.
      for (int s = 0; s < STAGES; ++s) {
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
      for (int w = pair; w < total && ok; w += num_pairs) {
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
          const uint32_t sA = base + stage * STAGE_BYTES;
          const uint64_t da = sw128_desc(sA);
          const uint64_t db = sw128_desc(sA + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes of K per step
            tc_mma(d, da + 2 * kk, db + 2 * kk, (kc | kk) != 0 ? 1u : 0u);
          tc_commit_both(empty_bar + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_both(accf_bar + 8 * acc);
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
      tc_commit_own(drain_bar);
      mbar_wait(drain_bar, 0, nullptr, DRAIN_LIMIT_NS);
    }
  } else {  // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row_in_cta = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t acce_c = map_to_cta(acce_bar, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = pair; w < total; w += num_pairs) {
      int mt, nt;
      raster(w, num_mt, a.n_tiles, mt, nt);
      const int e = a.tile_expert[mt];
      const int r = a.tile_row0[mt] + (int)rank * 128 + row_in_cta;
      const bool valid = r < a.offsets[e + 1];
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
      if (SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(t + c, g);
          tmem_ld16(t + 128 + c, u);
          tmem_wait_ld();
          if (valid && c < cols_left) {
            uint32_t p[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float h0 = silu(__uint_as_float(g[2 * q])) * __uint_as_float(u[2 * q]);
              const float h1 = silu(__uint_as_float(g[2 * q + 1])) * __uint_as_float(u[2 * q + 1]);
              p[q] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
            dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 256; c += 16) {
          uint32_t v[16];
          tmem_ld16(t + c, v);
          tmem_wait_ld();
          if (valid && c < cols_left) {
            uint32_t p[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              p[q] = pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
            dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_c + 8 * acc);
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 tensor [outer][mid][inner] (rank 3) or [outer][inner] (rank 2), boxes of
// 64 (inner) x 128 rows, 128-byte swizzle, out-of-range elements read as zero.
bool make_map(CUtensorMap* m, const void* ptr, int rank, uint64_t inner, uint64_t mid,
              uint64_t outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  cuuint32_t box[3] = {BK, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (rank == 2) dims[1] = outer;
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Clusters of two that can be resident at once (one CTA per SM): the grid size.
template <bool SWIGLU>
int grid_pairs() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_tc_kernel<SWIGLU>, &cfg) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = sms > 1 ? sms / 2 : 1;
  }
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

template <bool SWIGLU>
cudaError_t launch_t(const CUtensorMap& mA, const CUtensorMap& mB0, const CUtensorMap& mB1,
                     const TcArgs& t, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_tc_kernel<SWIGLU>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * grid_pairs<SWIGLU>(), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<SWIGLU>, mA, mB0, mB1, t);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_tc(const GroupedGemmArgs& a, cudaStream_t stream) {
  if (a.max_mtiles == 0 || a.A_rows == 0) return cudaSuccess;
  CUtensorMap mA, mB0, mB1;
  if (!make_map(&mA, a.A, 2, (uint64_t)a.K, 0, (uint64_t)a.A_rows)) return cudaErrorInvalidValue;
  if (!make_map(&mB0, a.B0, 3, (uint64_t)a.K, (uint64_t)a.n_cols, (uint64_t)a.N))
    return cudaErrorInvalidValue;
  if (!make_map(&mB1, a.swiglu ? a.B1 : a.B0, 3, (uint64_t)a.K, (uint64_t)a.n_cols, (uint64_t)a.N))
    return cudaErrorInvalidValue;
  TcArgs t;
  t.tile_expert = a.tile_expert;
  t.tile_row0 = a.tile_row0;
  t.offsets = a.offsets;
  t.num_mtiles = a.num_mtiles;
  t.out = static_cast<__nv_bfloat16*>(a.out);
  t.out_ld = a.n_cols;
  t.K = a.K;
  t.n_per_tile = a.swiglu ? 128 : 256;
  t.n_tiles = (a.n_cols + t.n_per_tile - 1) / t.n_per_tile;
  t.n_valid = a.n_cols;
  t.b1_row_off = a.swiglu ? 0 : 128;
  t.status = a.status;
  return a.swiglu ? launch_t<true>(mA, mB0, mB1, t, stream) : launch_t<false>(mA, mB0, mB1, t, stream);
}

}  // namespace moe
