// C-ABI entry points of the MoE forward library (declared in include/moe.h):
// argument checks, the workspace plan and the launch sequence. Every step of the
// layer runs in this library's kernels; the host only validates and enqueues.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

constexpr size_t kAlign = 256;
// The workspace starts with 256 bytes that must be zero before the first call
// (moe_workspace_init): the status word at offset 0 and the completion counters of the
// routing-decision kernel (offset 4) and of the rerouting kernel (offset 8), which
// those kernels return to zero themselves.
constexpr int kStatusBytes = 256;
constexpr size_t kDoneOffset = 4;
constexpr size_t kRerouteDoneOffset = 8;  // the rerouting kernel's completion counter

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Options of the *_ex entry points, with NULL read as the base layer.
struct Opts {
  int S = 0;                          // shared experts
  int act = MOE_ACT_SWIGLU;
  const uint8_t* valid = nullptr;     // [T] or null
  float* aux_kl = nullptr;
  float* aux_std2 = nullptr;
  bool reroute = false;
};

int read_opts(const moe_options* o, Opts* out) {
  Opts r;
  if (o != nullptr) {
    if (o->n_shared < 0 || o->n_shared > MOE_MAX_SHARED) return MOE_EINVAL;
    if (o->activation != MOE_ACT_SWIGLU && o->activation != MOE_ACT_GELU) return MOE_EINVAL;
    r.S = o->n_shared;
    r.act = o->activation;
    r.valid = o->valid_mask;
    r.aux_kl = o->aux_kl;
    r.aux_std2 = o->aux_std2;
    r.reroute = o->reroute != 0;
  }
  *out = r;
  return MOE_OK;
}

struct Plan {
  int T, H, N, k, F, dtype;
  int S;                  // shared experts (experts N..N+S-1 of the weight tensors)
  bool masked;            // a valid-token mask is given
  bool reroute;           // overflow rerouting (only with a capacity limit)
  bool fused;             // bf16 router GEMM and routing decisions in one launch
  float cf;               // capacity factor (<= 0: no limit)
  long long C;            // capacity without a mask, -1: no limit (an upper bound with one)
  int A;                  // T*k routing slots
  int A_cap;              // rows of the permuted buffers: kept routed slots + S*T
  int ksplit, chunks_per_split;
  int sel_tpw, n_sel_blocks;
  int max_mtiles[2];      // row tiles of 128 and of 256 rows, upper bounds
  bool pair1, pair2;      // GEMM1 / GEMM2 on 256-row tiles (CTA pairs), else 128-row
  bool pdl;               // kernels after the first launched as programmatic dependents
  size_t elem;
  size_t off_part, off_psum, off_blk, off_rank, off_idx, off_w, off_drop, off_counts,
      off_kept, off_offsets, off_tile_f[2], off_nmt, off_aux,
      off_cap, off_bvalid, off_vrank, off_bd2, off_rr_exp, off_rr_rank, off_rblk, off_slot_row,
      off_row_token, off_xp, off_h, off_ye, total;
};

int check_cfg(const moe_cfg* c) {
  if (c == nullptr) return MOE_EINVAL;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_EINVAL;
  if (c->T < 0 || c->H < 1 || c->N < 1 || c->k < 1 || c->F < 1 || c->k > c->N) return MOE_EINVAL;
  if (!(c->capacity_factor == c->capacity_factor)) return MOE_EINVAL;  // NaN
  if (c->N > 256 || c->k > 32 || c->H % 64 != 0 || c->F % 64 != 0) return MOE_EUNSUPPORTED;
  if ((long long)c->T * c->k > (1ll << 30)) return MOE_EUNSUPPORTED;
  return MOE_OK;
}

long long capacity_of(const moe_cfg* c) {
  if (!(c->capacity_factor > 0.0f)) return -1;
  const double cap = ceil((double)c->capacity_factor * (double)c->T * (double)c->k / (double)c->N);
  const double slots = (double)c->T * (double)c->k;
  return cap >= slots ? (long long)slots : (long long)cap;  // an expert never holds more
}

Plan make_plan(const moe_cfg* c, const Opts& o) {
  Plan p;
  memset(&p, 0, sizeof(p));
  p.T = c->T; p.H = c->H; p.N = c->N; p.k = c->k; p.F = c->F; p.dtype = c->dtype;
  p.S = o.S;
  p.masked = o.valid != nullptr;
  p.reroute = o.reroute && c->capacity_factor > 0.0f;
  p.cf = c->capacity_factor;
  p.C = capacity_of(c);  // with a mask the call's C (from T_valid <= T) is no larger
  p.A = c->T * c->k;
  long long cap_rows = p.A;
  if (p.C >= 0 && (long long)p.N * p.C < cap_rows) cap_rows = (long long)p.N * p.C;
  cap_rows += (long long)p.S * p.T;
  p.A_cap = (int)cap_rows;
  p.elem = c->dtype == MOE_BF16 ? 2 : 4;
  // Router split over H: keep about two blocks per SM when T is small.
  const int nblk = (p.T + ROUTER_TOKENS - 1) / ROUTER_TOKENS;
  const int nchunk = p.H / ROUTER_KC;
  int ksplit = nblk > 0 ? (296 + nblk - 1) / nblk : 1;
  if (ksplit > 16) ksplit = 16;
  if (ksplit > nchunk) ksplit = nchunk;
  if (ksplit < 1) ksplit = 1;
  p.chunks_per_split = (nchunk + ksplit - 1) / ksplit;
  p.ksplit = (nchunk + p.chunks_per_split - 1) / p.chunks_per_split;
  // routing decisions: one token per warp at a time; about 600 blocks at most, so
  // the last block's scan over the blocks stays short
  p.sel_tpw = p.T / (SELECT_WARPS * 600) > 1 ? p.T / (SELECT_WARPS * 600) : 1;
  // bf16 router: with at least 32 tiles of 128 tokens, one fused launch (router GEMM
  // and routing decisions, no split of K: its logits, for rerouting, are one "split";
  // the rerouting kernel and dispatch use its 128-token blocks, 32 warps x 4 tokens).
  // Fewer tiles leave too few SMs streaming x, so the tensor-core router splits K over
  // the GPU and the routing decisions follow in their own launch.
  p.fused = p.dtype == MOE_BF16 && (p.T + ROUTE_FUSED_TOKENS - 1) / ROUTE_FUSED_TOKENS >= 32;
  if (p.fused) {
    p.ksplit = 1;
    p.sel_tpw = ROUTE_FUSED_TOKENS / SELECT_WARPS;
  } else if (p.dtype == MOE_BF16) {
    int kcps = 0;
    router_tc_split(p.T, p.H, &p.ksplit, &kcps);
  }
  p.n_sel_blocks = (p.T + SELECT_WARPS * p.sel_tpw - 1) / (SELECT_WARPS * p.sel_tpw);
  p.max_mtiles[0] = (p.A_cap + TILE_ROWS_1 - 1) / TILE_ROWS_1 + p.N + p.S;
  p.max_mtiles[1] = (p.A_cap + TILE_ROWS_2 - 1) / TILE_ROWS_2 + p.N + p.S;
  // Expert GEMM tile shapes (see choose_tiles); this default holds without a bias.
  p.pair1 = p.pair2 = (long long)p.T * (p.k + p.S) >= 1024ll * (p.N + p.S);
  p.pdl = p.dtype == MOE_BF16;

  size_t cur = kStatusBytes;
  auto take = [&](size_t bytes) {
    const size_t o = cur;
    cur = align_up(cur + (bytes > 0 ? bytes : 1), kAlign);
    return o;
  };
  const size_t T = p.T, N = p.N, A = p.A, Ac = p.A_cap, NS = (size_t)p.N + p.S;
  p.off_part = take((size_t)p.ksplit * T * N * 4);
  p.off_psum = take((size_t)p.n_sel_blocks * N * 4);
  p.off_blk = take((size_t)p.n_sel_blocks * N * 4);
  p.off_rank = take(A * 4);
  p.off_idx = take(A * 4);
  p.off_w = take(A * 4);
  p.off_drop = take(A);
  p.off_counts = take(NS * 4);
  p.off_kept = take(NS * 4);
  p.off_offsets = take((NS + 1) * 4);
  for (int tb = 0; tb < 2; ++tb) p.off_tile_f[tb] = take((NS + 1) * 4);
  p.off_nmt = take(8);
  p.off_aux = take(4);
  p.off_cap = take(4);
  p.off_bvalid = take((size_t)p.n_sel_blocks * 4);
  p.off_vrank = take(p.masked && p.S > 0 ? T * 4 : 0);
  p.off_bd2 = take((size_t)p.n_sel_blocks * 4);
  p.off_rr_exp = take(p.reroute ? A * 4 : 0);
  p.off_rr_rank = take(p.reroute ? A * 4 : 0);
  p.off_rblk = take(p.reroute ? (size_t)p.n_sel_blocks * N * 4 : 0);
  p.off_slot_row = take(T * (size_t)(p.k + p.S) * 4);
  p.off_row_token = take(Ac * 4);
  p.off_xp = take(Ac * p.H * p.elem);
  p.off_h = take(Ac * p.F * p.elem);
  p.off_ye = take(Ac * p.H * p.elem);
  p.total = cur;
  return p;
}

// Expected rows one expert GEMM computes, over all experts, with tiles of m rows: a
// routed expert's slot count taken as Normal(mu, sigma^2), the binomial count of
// uniform routing (mu = T*k/N, sigma^2 = mu*(1 - 1/N)), limited by the capacity;
// a shared expert has T rows.
double expected_rows(const Plan& p, int m) {
  const double mu = (double)p.T * p.k / p.N;
  const double sigma = sqrt(mu * (1.0 - 1.0 / p.N));
  double num = 0.0, den = 0.0;
  for (int i = -320; i <= 320; ++i) {  // z in [-4, 4] in steps of 1/80
    const double z = i / 80.0;
    double c = mu + z * sigma;
    if (c < 0.0) c = 0.0;
    if (p.C >= 0 && c > (double)p.C) c = (double)p.C;
    const double w = exp(-0.5 * z * z);
    num += w * ceil(c / m) * m;
    den += w;
  }
  const double shared = (double)p.S * ceil((double)p.T / m) * m;
  return p.N * (num / den) + shared;
}

// Tile shape of each expert GEMM. CTA pairs (256-row tiles) stage a third fewer
// bytes per SM for the same MMA work, so their load pipeline hides more latency: on
// B300 they process computed rows about 1.17x faster than single CTAs (128-row
// tiles), but every expert's last tile is padded to 256 rows. GEMM2 has few column
// tiles (H/256), so wave quantisation decides it: pairs only from 1024 expected rows
// per expert. GEMM1 also takes pairs from 512 expected rows per expert when the pair
// computes at most 12% more rows than single CTAs under the uniform-routing count
// model; with a router bias the counts are skewed in ways the host cannot see, so
// GEMM1 keeps the 1024-row rule there.
void choose_tiles(Plan& p, bool has_bias) {
  const long long rows = (long long)p.T * (p.k + p.S), per = 1024ll * (p.N + p.S);
  p.pair2 = rows >= per;
  p.pair1 = p.pair2;
  if (!p.pair1 && !has_bias && (long long)p.T * p.k >= 512ll * p.N)
    p.pair1 = expected_rows(p, TILE_ROWS_2) <= 1.12 * expected_rows(p, TILE_ROWS_1);
}

int device_check() {
  static std::atomic<int> ok_dev[64];  // 0 unknown, 1 sm_103, -1 other
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ECUDA;
  if (dev >= 0 && dev < 64) {
    const int known = ok_dev[dev].load(std::memory_order_relaxed);
    if (known != 0) return known > 0 ? MOE_OK : MOE_ENODEVICE;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ECUDA;
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < 64) ok_dev[dev].store(ok ? 1 : -1, std::memory_order_relaxed);
  return ok ? MOE_OK : MOE_ENODEVICE;
}

#define MOE_TRY(expr)                                \
  do {                                               \
    if ((expr) != cudaSuccess) return MOE_ECUDA;     \
  } while (0)

struct Outs {
  int32_t* idx;
  float* w;
  float* aux;
  uint8_t* drop;
  int32_t* counts;
  int32_t* kept;
};

// Shared front half: router, capacity, dispatch. `copy` gathers x into xp.
int run_route(const Plan& p, const Opts& op, const void* x, const void* w_router,
              const float* bias, const Outs& o, uint8_t* ws, bool copy, cudaStream_t s,
              cudaEvent_t* ev) {
  auto rec = [&](int i) {
    if (ev != nullptr) cudaEventRecord(ev[i], s);
  };
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* part = reinterpret_cast<float*>(ws + p.off_part);
  const bool fused = p.fused;
  rec(0);
  if (p.dtype == MOE_BF16 && !fused)
    MOE_TRY(launch_router_logits_tc(x, w_router, part, p.T, p.H, p.N, status, s, false));
  else if (!fused)
    MOE_TRY(launch_router_logits(p.dtype, x, w_router, part, p.T, p.H, p.N, p.ksplit,
                                 p.chunks_per_split, s));
  rec(1);  // fused: the router runs inside the routing-decision stage
  SelectArgs sa;
  sa.part = part;
  sa.ksplit = p.ksplit;
  sa.bias = bias;
  sa.T = p.T; sa.N = p.N; sa.k = p.k;
  sa.S = p.S;
  sa.valid = op.valid;
  sa.vrank = reinterpret_cast<int32_t*>(ws + p.off_vrank);
  sa.blk_valid = reinterpret_cast<int32_t*>(ws + p.off_bvalid);
  sa.blk_d2 = reinterpret_cast<float*>(ws + p.off_bd2);
  sa.cap = reinterpret_cast<int32_t*>(ws + p.off_cap);
  sa.C = p.C;
  sa.cf = (double)p.cf;
  sa.aux_kl = op.aux_kl;
  sa.aux_std2 = op.aux_std2;
  sa.tpw = p.sel_tpw;
  sa.idx = o.idx;
  sa.w = o.w;
  sa.slot_rank = reinterpret_cast<int32_t*>(ws + p.off_rank);
  sa.blk_counts = reinterpret_cast<int32_t*>(ws + p.off_blk);
  sa.blk_psum = reinterpret_cast<float*>(ws + p.off_psum);
  sa.done = reinterpret_cast<unsigned*>(ws + kDoneOffset);
  sa.counts = reinterpret_cast<int32_t*>(ws + p.off_counts);
  sa.kept = reinterpret_cast<int32_t*>(ws + p.off_kept);
  sa.offsets = reinterpret_cast<int32_t*>(ws + p.off_offsets);
  for (int tb = 0; tb < 2; ++tb) {
    sa.num_mtiles[tb] = reinterpret_cast<int32_t*>(ws + p.off_nmt) + tb;
    sa.tile_first[tb] = reinterpret_cast<int32_t*>(ws + p.off_tile_f[tb]);
  }
  sa.aux = o.aux;
  sa.user_counts = o.counts;
  sa.user_kept = o.kept;
  if (fused)  // the forward's first kernel: not a dependent launch
    MOE_TRY(launch_route_fused(sa, x, w_router, p.H, p.reroute ? part : nullptr, status, s,
                               false));
  else
    MOE_TRY(launch_route_select(sa, p.n_sel_blocks, s, p.pdl));
  RerouteArgs ra;
  if (p.reroute) {
    ra.part = part;
    ra.ksplit = p.ksplit;
    ra.bias = fused ? nullptr : bias;  // the fused kernel's logits include the bias
    ra.T = p.T; ra.N = p.N; ra.k = p.k; ra.S = p.S;
    ra.tpw = p.sel_tpw;
    ra.idx = o.idx;
    ra.slot_rank = sa.slot_rank;
    ra.blk_base = sa.blk_counts;
    ra.counts = sa.counts;
    ra.kept = sa.kept;
    ra.cap = sa.cap;
    ra.rr_exp = reinterpret_cast<int32_t*>(ws + p.off_rr_exp);
    ra.rr_rank = reinterpret_cast<int32_t*>(ws + p.off_rr_rank);
    ra.rblk = reinterpret_cast<int32_t*>(ws + p.off_rblk);
    ra.done = reinterpret_cast<unsigned*>(ws + kRerouteDoneOffset);
    ra.offsets = sa.offsets;
    for (int tb = 0; tb < 2; ++tb) {
      ra.num_mtiles[tb] = sa.num_mtiles[tb];
      ra.tile_first[tb] = sa.tile_first[tb];
    }
    ra.user_kept = o.kept;
    MOE_TRY(launch_reroute(ra, p.n_sel_blocks, s, p.pdl));
  }
  rec(2);
  DispatchArgs da;
  da.idx = o.idx;
  da.slot_rank = sa.slot_rank;
  da.blk_base = sa.blk_counts;
  da.tokens_per_block = SELECT_WARPS * p.sel_tpw;
  da.offsets = sa.offsets;
  da.cap = sa.cap;
  da.C = p.C;
  da.T = p.T; da.k = p.k; da.N = p.N; da.H = p.H;
  da.S = p.S;
  da.valid = op.valid;
  da.vrank = sa.vrank;
  da.blk_vbase = sa.blk_valid;
  da.rr_exp = p.reroute ? ra.rr_exp : nullptr;
  da.rr_rank = p.reroute ? ra.rr_rank : nullptr;
  da.rr_base = p.reroute ? ra.rblk : nullptr;
  da.counts = sa.counts;
  da.A_cap = p.A_cap;
  da.x = x;
  da.xp = ws + p.off_xp;
  da.drop = o.drop;
  da.slot_row = reinterpret_cast<int32_t*>(ws + p.off_slot_row);
  da.row_token = reinterpret_cast<int32_t*>(ws + p.off_row_token);
  da.status = status;
  MOE_TRY(launch_dispatch(p.dtype, copy, da, s, p.pdl));
  rec(3);
  return MOE_OK;
}

int run_experts(const Plan& p, const Opts& op, const void* w1, const void* w3, const void* w2,
                void* out, const Outs& o, uint8_t* ws, cudaStream_t s, cudaEvent_t* ev) {
  auto rec = [&](int i) {
    if (ev != nullptr) cudaEventRecord(ev[i], s);
  };
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  GroupedGemmArgs g;
  g.A = ws + p.off_xp;
  g.A_rows = p.A_cap;
  g.B0 = w1;
  g.B1 = op.act == MOE_ACT_SWIGLU ? w3 : nullptr;
  g.out = ws + p.off_h;
  g.K = p.H;
  g.n_cols = p.F;
  g.N = p.N + p.S;
  g.epi = op.act == MOE_ACT_GELU ? EPI_GELU : EPI_SWIGLU;
  // float32 layers run on CUDA cores over the 128-row table
  int tb = (p.dtype == MOE_BF16 && p.pair1) ? 1 : 0;
  g.pair = tb == 1;
  g.offsets = reinterpret_cast<const int32_t*>(ws + p.off_offsets);
  g.num_mtiles = reinterpret_cast<const int32_t*>(ws + p.off_nmt) + tb;
  g.tile_first = reinterpret_cast<const int32_t*>(ws + p.off_tile_f[tb]);
  g.max_mtiles = p.max_mtiles[tb];
  g.status = status;
  if (p.dtype == MOE_BF16) MOE_TRY(launch_grouped_gemm_tc(g, s, p.pdl));
  else MOE_TRY(launch_grouped_gemm_simt(g, s));
  rec(4);
  tb = (p.dtype == MOE_BF16 && p.pair2) ? 1 : 0;
  g.pair = tb == 1;
  g.num_mtiles = reinterpret_cast<const int32_t*>(ws + p.off_nmt) + tb;
  g.tile_first = reinterpret_cast<const int32_t*>(ws + p.off_tile_f[tb]);
  g.max_mtiles = p.max_mtiles[tb];
  g.A = ws + p.off_h;
  g.B0 = w2;
  g.B1 = nullptr;
  g.out = ws + p.off_ye;
  g.K = p.F;
  g.n_cols = p.H;
  g.epi = EPI_PLAIN;
  if (p.dtype == MOE_BF16) MOE_TRY(launch_grouped_gemm_tc(g, s, p.pdl));
  else MOE_TRY(launch_grouped_gemm_simt(g, s));
  rec(5);
  MOE_TRY(launch_combine(p.dtype, ws + p.off_ye,
                         reinterpret_cast<const int32_t*>(ws + p.off_slot_row), o.w, p.T, p.k,
                         p.S, p.H, out, s, p.pdl));
  rec(6);
  return MOE_OK;
}

int check_ws(const Plan& p, void* ws, size_t ws_bytes) {
  if (ws == nullptr || !aligned(ws, kAlign) || ws_bytes < p.total) return MOE_EWORKSPACE;
  return MOE_OK;
}

// Options that fit the layer: slot rows of the shared experts stay within the limit
// on routing slots.
int check_opts(const moe_cfg* c, const Opts& o) {
  if ((long long)c->T * (c->k + o.S) > (1ll << 30)) return MOE_EUNSUPPORTED;
  return MOE_OK;
}

// T = 0: nothing to route; the losses and the counts are zero.
int empty_batch(const Plan& p, const Opts& op, float* aux, int32_t* counts, int32_t* kept,
                cudaStream_t s, cudaEvent_t* ev) {
  if (ev != nullptr)
    for (int i = 0; i <= MOE_NUM_STAGES; ++i) cudaEventRecord(ev[i], s);
  if (aux != nullptr) MOE_TRY(cudaMemsetAsync(aux, 0, sizeof(float), s));
  if (op.aux_kl != nullptr) MOE_TRY(cudaMemsetAsync(op.aux_kl, 0, sizeof(float), s));
  if (op.aux_std2 != nullptr) MOE_TRY(cudaMemsetAsync(op.aux_std2, 0, sizeof(float), s));
  if (counts != nullptr) MOE_TRY(cudaMemsetAsync(counts, 0, p.N * sizeof(int32_t), s));
  if (kept != nullptr) MOE_TRY(cudaMemsetAsync(kept, 0, p.N * sizeof(int32_t), s));
  return MOE_OK;
}

int forward_impl(const moe_cfg* cfg, const moe_options* opts, const void* x,
                 const void* w_router, const float* bias, const void* w1, const void* w3,
                 const void* w2, void* out, int32_t* topk_idx, float* topk_w, float* aux_loss,
                 uint8_t* drop_mask, int32_t* expert_counts, int32_t* kept_counts,
                 void* workspace, size_t workspace_bytes, void* stream,
                 void* const* stage_events) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  Opts op;
  rc = read_opts(opts, &op);
  if (rc != MOE_OK) return rc;
  rc = check_opts(cfg, op);
  if (rc != MOE_OK) return rc;
  // x and out hold T rows: with T = 0 they may be NULL (an empty tensor's address).
  if (w_router == nullptr || w1 == nullptr || w2 == nullptr ||
      (op.act == MOE_ACT_SWIGLU && w3 == nullptr) ||
      (cfg->T > 0 && (x == nullptr || out == nullptr)))
    return MOE_EINVAL;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(w1, 16) || !aligned(w3, 16) ||
      !aligned(w2, 16) || !aligned(out, 16) || !aligned(bias, 4) || !aligned(topk_idx, 4) ||
      !aligned(topk_w, 4) || !aligned(aux_loss, 4) || !aligned(expert_counts, 4) ||
      !aligned(kept_counts, 4) || !aligned(op.aux_kl, 4) || !aligned(op.aux_std2, 4))
    return MOE_EALIGN;
  Plan p = make_plan(cfg, op);
  choose_tiles(p, bias != nullptr);
  rc = check_ws(p, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  rc = device_check();
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t* ev = stage_events ? reinterpret_cast<cudaEvent_t*>(const_cast<void**>(stage_events))
                                 : nullptr;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (p.T == 0) return empty_batch(p, op, aux_loss, expert_counts, kept_counts, s, ev);
  Outs o;
  o.idx = topk_idx ? topk_idx : reinterpret_cast<int32_t*>(ws + p.off_idx);
  o.w = topk_w ? topk_w : reinterpret_cast<float*>(ws + p.off_w);
  o.aux = aux_loss ? aux_loss : reinterpret_cast<float*>(ws + p.off_aux);
  o.drop = drop_mask ? drop_mask : ws + p.off_drop;
  o.counts = expert_counts;
  o.kept = kept_counts;
  rc = run_route(p, op, x, w_router, bias, o, ws, true, s, ev);
  if (rc != MOE_OK) return rc;
  return run_experts(p, op, w1, w3, w2, out, o, ws, s, ev);
}

int route_impl(const moe_cfg* cfg, const moe_options* opts, const void* x,
               const void* w_router, const float* router_bias, int32_t* topk_idx,
               float* topk_w, float* aux_loss, uint8_t* drop_mask, int32_t* expert_counts,
               int32_t* kept_counts, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  Opts op;
  rc = read_opts(opts, &op);
  if (rc != MOE_OK) return rc;
  rc = check_opts(cfg, op);
  if (rc != MOE_OK) return rc;
  if (w_router == nullptr || aux_loss == nullptr ||
      (cfg->T > 0 && (x == nullptr || topk_idx == nullptr || topk_w == nullptr ||
                      drop_mask == nullptr)))
    return MOE_EINVAL;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(router_bias, 4) ||
      !aligned(topk_idx, 4) || !aligned(topk_w, 4) || !aligned(aux_loss, 4) ||
      !aligned(expert_counts, 4) || !aligned(kept_counts, 4) || !aligned(op.aux_kl, 4) ||
      !aligned(op.aux_std2, 4))
    return MOE_EALIGN;
  const Plan p = make_plan(cfg, op);
  rc = check_ws(p, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  rc = device_check();
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (p.T == 0) return empty_batch(p, op, aux_loss, expert_counts, kept_counts, s, nullptr);
  Outs o{topk_idx, topk_w, aux_loss, drop_mask, expert_counts, kept_counts};
  return run_route(p, op, x, w_router, router_bias, o, ws, false, s, nullptr);
}

// Routing scratch for callers that cannot allocate device memory (see
// moe_route_static). Every GPU that loads this library holds this array until the
// process exits; all calls share it.
constexpr size_t kStaticScratchBytes = MOE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_route_scratch[kStaticScratchBytes];

// Device address of g_route_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached. Two threads making the first call on
// one device may both look it up; they store the same address.
int static_scratch(uint8_t** out) {
  static std::atomic<void*> addr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ECUDA;
  void* a = addr[dev].load(std::memory_order_acquire);
  if (a == nullptr) {
    if (cudaGetSymbolAddress(&a, g_route_scratch) != cudaSuccess || a == nullptr)
      return MOE_ECUDA;
    addr[dev].store(a, std::memory_order_release);
  }
  *out = static_cast<uint8_t*>(a);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_cfg* cfg) { return moe_workspace_size_ex(cfg, nullptr); }

size_t moe_workspace_size_ex(const moe_cfg* cfg, const moe_options* opts) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  Opts op;
  if (read_opts(opts, &op) != MOE_OK || check_opts(cfg, op) != MOE_OK) return 0;
  return make_plan(cfg, op).total;
}

int moe_describe(const moe_cfg* cfg, const moe_options* opts, int has_bias, moe_plan* plan) {
  if (plan == nullptr) return MOE_EINVAL;
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  Opts op;
  rc = read_opts(opts, &op);
  if (rc != MOE_OK) return rc;
  rc = check_opts(cfg, op);
  if (rc != MOE_OK) return rc;
  Plan p = make_plan(cfg, op);
  choose_tiles(p, has_bias != 0);
  const bool tc = p.dtype == MOE_BF16;
  plan->fused_routing = p.fused ? 1 : 0;
  plan->routing_block = SELECT_WARPS * p.sel_tpw;
  plan->router_ksplit = p.ksplit;
  plan->gemm1_tile_rows = tc && p.pair1 ? TILE_ROWS_2 : TILE_ROWS_1;
  plan->gemm2_tile_rows = tc && p.pair2 ? TILE_ROWS_2 : TILE_ROWS_1;
  // routing (one kernel fused, else router + decisions), rerouting, dispatch, two
  // expert GEMMs, combine: the launches run_route and run_experts make
  plan->launches = (p.fused ? 1 : 2) + (p.reroute ? 1 : 0) + 1 + 2 + 1;
  plan->capacity = p.C;
  plan->workspace_bytes = (int64_t)p.total;
  // the routing kernel the forward launches: its finish and its threads per block
  const bool plain = op.valid == nullptr && op.aux_kl == nullptr && op.aux_std2 == nullptr;
  const int nblk = p.fused ? (p.T + ROUTE_FUSED_TOKENS - 1) / ROUTE_FUSED_TOKENS : p.n_sel_blocks;
  plan->routing_threads = p.fused ? route_fused_threads(p.N) : SELECT_WARPS * 32;
  plan->routing_warp_finish =
      warp_finish_fits(p.N, nblk, plain,
                       p.fused ? FUSED_WARP_FINISH_ROWS : SELECT_WARP_FINISH_ROWS) &&
              !(p.fused && plan->routing_threads != 256)
          ? 1
          : 0;
  return MOE_OK;
}

int moe_capacity(const moe_cfg* cfg, int64_t* capacity) {
  if (capacity == nullptr) return MOE_EINVAL;
  const int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  *capacity = capacity_of(cfg);
  return MOE_OK;
}

int moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || !aligned(workspace, kAlign) || workspace_bytes < (size_t)kStatusBytes)
    return MOE_EWORKSPACE;
  const int rc = device_check();
  if (rc != MOE_OK) return rc;
  MOE_TRY(cudaMemsetAsync(workspace, 0, kStatusBytes, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_route(const moe_cfg* cfg, const void* x, const void* w_router, const float* router_bias,
              int32_t* topk_idx, float* topk_w, float* aux_loss, uint8_t* drop_mask,
              int32_t* expert_counts, int32_t* kept_counts, void* workspace,
              size_t workspace_bytes, void* stream) {
  return route_impl(cfg, nullptr, x, w_router, router_bias, topk_idx, topk_w, aux_loss,
                    drop_mask, expert_counts, kept_counts, workspace, workspace_bytes, stream);
}

int moe_route_ex(const moe_cfg* cfg, const moe_options* opts, const void* x,
                 const void* w_router, const float* router_bias, int32_t* topk_idx,
                 float* topk_w, float* aux_loss, uint8_t* drop_mask, int32_t* expert_counts,
                 int32_t* kept_counts, void* workspace, size_t workspace_bytes, void* stream) {
  return route_impl(cfg, opts, x, w_router, router_bias, topk_idx, topk_w, aux_loss, drop_mask,
                    expert_counts, kept_counts, workspace, workspace_bytes, stream);
}

int moe_route_static(const moe_cfg* cfg, const void* x, const void* w_router,
                     const float* router_bias, int32_t* topk_idx, float* topk_w, float* aux_loss,
                     uint8_t* drop_mask, int32_t* expert_counts, int32_t* kept_counts,
                     void* stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (w_router == nullptr || aux_loss == nullptr ||
      (cfg->T > 0 && (x == nullptr || topk_idx == nullptr || topk_w == nullptr ||
                      drop_mask == nullptr)))
    return MOE_EINVAL;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(router_bias, 4) ||
      !aligned(topk_idx, 4) || !aligned(topk_w, 4) || !aligned(aux_loss, 4) ||
      !aligned(expert_counts, 4) || !aligned(kept_counts, 4))
    return MOE_EALIGN;
  const Opts op;
  const Plan p = make_plan(cfg, op);
  // The routing half uses the workspace prefix that ends where the expert buffers
  // begin; it must fit the static array.
  if (p.off_xp > kStaticScratchBytes) return MOE_EUNSUPPORTED;
  rc = device_check();
  if (rc != MOE_OK) return rc;
  uint8_t* ws = nullptr;
  rc = static_scratch(&ws);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word must start at 0.
  MOE_TRY(cudaMemsetAsync(ws, 0, kStatusBytes, s));
  if (p.T == 0) return empty_batch(p, op, aux_loss, expert_counts, kept_counts, s, nullptr);
  Outs o{topk_idx, topk_w, aux_loss, drop_mask, expert_counts, kept_counts};
  return run_route(p, op, x, w_router, router_bias, o, ws, false, s, nullptr);
}

int moe_forward(const moe_cfg* cfg, const void* x, const void* w_router, const float* router_bias,
                const void* w1, const void* w3, const void* w2, void* out, int32_t* topk_idx,
                float* topk_w, float* aux_loss, uint8_t* drop_mask, int32_t* expert_counts,
                int32_t* kept_counts, void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(cfg, nullptr, x, w_router, router_bias, w1, w3, w2, out, topk_idx, topk_w,
                      aux_loss, drop_mask, expert_counts, kept_counts, workspace,
                      workspace_bytes, stream, nullptr);
}

int moe_forward_timed(const moe_cfg* cfg, const void* x, const void* w_router,
                      const float* router_bias, const void* w1, const void* w3, const void* w2,
                      void* out, int32_t* topk_idx, float* topk_w, float* aux_loss,
                      uint8_t* drop_mask, int32_t* expert_counts, int32_t* kept_counts,
                      void* workspace, size_t workspace_bytes, void* stream,
                      void* const* stage_events) {
  return forward_impl(cfg, nullptr, x, w_router, router_bias, w1, w3, w2, out, topk_idx, topk_w,
                      aux_loss, drop_mask, expert_counts, kept_counts, workspace,
                      workspace_bytes, stream, stage_events);
}

int moe_forward_ex(const moe_cfg* cfg, const moe_options* opts, const void* x,
                   const void* w_router, const float* router_bias, const void* w1,
                   const void* w3, const void* w2, void* out, int32_t* topk_idx, float* topk_w,
                   float* aux_loss, uint8_t* drop_mask, int32_t* expert_counts,
                   int32_t* kept_counts, void* workspace, size_t workspace_bytes, void* stream,
                   void* const* stage_events) {
  return forward_impl(cfg, opts, x, w_router, router_bias, w1, w3, w2, out, topk_idx, topk_w,
                      aux_loss, drop_mask, expert_counts, kept_counts, workspace,
                      workspace_bytes, stream, stage_events);
}

namespace moe {
namespace {
// Synchronise `stream`, then read and clear the status word at `word_addr`.
int read_status(void* word_addr, cudaStream_t s, uint32_t* bits) {
  uint32_t word = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ECUDA;
  if (cudaMemcpy(&word, word_addr, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ECUDA;
  if (bits != nullptr) *bits = word;
  if (word != 0) {
    if (cudaMemset(word_addr, 0, sizeof(word)) != cudaSuccess) return MOE_ECUDA;
    return MOE_EDEVICE;
  }
  return MOE_OK;
}
}  // namespace
}  // namespace moe

int moe_get_status(void* workspace, size_t workspace_bytes, void* stream, uint32_t* bits) {
  if (workspace == nullptr || !aligned(workspace, kAlign) || workspace_bytes < (size_t)kStatusBytes)
    return MOE_EWORKSPACE;
  return read_status(workspace, static_cast<cudaStream_t>(stream), bits);
}

int moe_get_status_static(void* stream, uint32_t* bits) {
  int rc = device_check();
  if (rc != MOE_OK) return rc;
  uint8_t* ws = nullptr;
  rc = static_scratch(&ws);
  if (rc != MOE_OK) return rc;
  return read_status(ws, static_cast<cudaStream_t>(stream), bits);
}

const char* moe_strerror(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument";
    case MOE_EUNSUPPORTED: return "layer shape outside the supported range";
    case MOE_EWORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_EALIGN: return "tensor pointer misaligned";
    case MOE_ECUDA: return "CUDA runtime error";
    case MOE_EDEVICE: return "a kernel reported a device-side failure";
    case MOE_ENODEVICE: return "current device is not an sm_103 GPU";
    default: return "unknown status";
  }
}

}  // extern "C"
