/*
 * moe.h -- C ABI of the B300 (sm_103a) forward pass of one top-k routed
 * Mixture-of-Experts FFN layer.
 *
 * The layer, as the pages state it:
 *   logits = x W_r^T (+ b)                  router: a small linear layer hidden -> N
 *   idx, w = top-k(logits), softmax over the k selected logits
 *   aux    = N * sum_e f_e * P_e            load-balancing loss
 *   C      = ceil(CF * T * k / N)           per-expert capacity; overflow is dropped
 *   y[t]   = sum over kept slots s of w[t,s] * W2_e (silu(W1_e x_t) * (W3_e x_t))
 * Sources: cf-1.com/news/5914943 sections 2.1 (router, top-k, softmax, weighted
 * sum) and 2.3 (aux loss, capacity note); 2kiu.com/news/2885792 sections 2.2
 * (SwiGLU experts, capacity factor) and 3.1 (hard top-k with capacity, first
 * tokens kept); hotelren.com/news/3071227 section 4.1 (router returns indices,
 * weights, mask); 2kiu.com/news/2885792 section 5.3 (equal logits ordered by
 * ascending expert id).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device, row-major
 *    and densely packed, 16-byte aligned. The caller owns and allocates every
 *    buffer, including the workspace; the library allocates no device memory and
 *    keeps no state between calls.
 *  - Element type of x, w_router, w1, w3, w2, out: float32 (MOE_F32) or bf16
 *    (MOE_BF16) as cfg->dtype says. router_bias is always float32.
 *  - Shapes: x [T,H]; w_router [N,H]; router_bias [N]; w1, w3 [N,F,H] and
 *    w2 [N,H,F]; every weight in nn.Linear [out,in] orientation (the router's
 *    as the pages' nn.Linear(hidden, num_experts), the experts' per expert); out [T,H];
 *    topk_idx [T,k] int32; topk_w [T,k] float32; drop_mask [T,k] uint8
 *    (1 = slot dropped by capacity); expert_counts, kept_counts [N] int32;
 *    aux_loss [1] float32.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). A return of MOE_OK means the work was enqueued. Arguments are
 *    checked on the host before anything is enqueued; a failed argument check
 *    enqueues nothing and touches no CUDA API (the device check, which asks the
 *    runtime for the current device's compute capability, comes after them).
 *  - Kernels report device-side failures (a bounded wait that gave up, an index
 *    out of range) by OR-ing bits into a status word inside the workspace;
 *    moe_get_status() reads and clears it.
 *  - Calls sharing one workspace must not overlap on the GPU (use one stream).
 *  - Supported: 1 <= k <= min(N, 32), 1 <= N <= 256, T >= 0, H and F multiples
 *    of 64. The library is built for sm_103a only.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_EINVAL = 1,        /* NULL required pointer, negative size, k > N, bad dtype */
  MOE_EUNSUPPORTED = 2,  /* a valid layer outside the supported range above */
  MOE_EWORKSPACE = 3,    /* workspace NULL, misaligned or smaller than moe_workspace_size */
  MOE_EALIGN = 4,        /* a tensor pointer that is not 16-byte aligned */
  MOE_ECUDA = 5,         /* a CUDA runtime call or a kernel launch failed */
  MOE_EDEVICE = 6,       /* a kernel set the workspace status word */
  MOE_ENODEVICE = 7      /* the current device is not an sm_103 GPU */
};

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* One layer instance. capacity_factor <= 0 means no capacity limit. */
typedef struct {
  int32_t T;                 /* tokens (batch * seq_len) */
  int32_t H;                 /* hidden size */
  int32_t N;                 /* routed experts */
  int32_t k;                 /* experts per token */
  int32_t F;                 /* SwiGLU inner width of one expert */
  float capacity_factor;     /* CF of C = ceil(CF*T*k/N) */
  int32_t dtype;             /* moe_dtype */
} moe_cfg;

/* Number of stages moe_forward_timed() brackets with events. */
#define MOE_NUM_STAGES 6

/*
 * Bytes of device workspace moe_route / moe_forward need for `cfg`; 0 if cfg is
 * invalid or unsupported. Pure host function; the size grows linearly in T*k*(H+F).
 */
size_t moe_workspace_size(const moe_cfg* cfg);

/*
 * Per-expert capacity C = ceil(CF*T*k/N) (2kiu.com/news/2885792 section 3.1 keeps
 * the first C tokens of each expert; cf-1.com/news/5914943 section 2.3 sends the
 * overflow to the residual). CF is the float32 value of cfg->capacity_factor and
 * the product is evaluated in double as ((CF*T)*k)/N. Writes -1 when there is no
 * limit. Pure host function. Returns MOE_OK or MOE_EINVAL.
 */
int moe_capacity(const moe_cfg* cfg, int64_t* capacity);

/*
 * Zero the workspace's first 256 bytes: the status word and a completion counter
 * that the kernels keep at zero between calls. Call once after allocating a
 * workspace whose contents are unknown (a zero-filled allocation needs no call).
 * Asynchronous on `stream`.
 */
int moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Routing half of the layer (hotelren.com/news/3071227 section 4.1: the router
 * returns expert indices, weights and a mask):
 *   topk_idx[t,s]  the s-th largest logit's expert (ties: lower expert id first)
 *   topk_w[t,s]    softmax over the k selected logits
 *   aux_loss[0]    N * sum_e (counts_e/(T*k)) * (sum_t P[t,e] / T), P the softmax
 *                  over all N logits, counts taken before capacity (T = 0 gives 0)
 *   drop_mask[t,s] 1 when the slot's rank among the expert's slots, in token order,
 *                  is >= C
 *   expert_counts  slots per expert before capacity (optional, NULL ok)
 *   kept_counts    slots per expert after capacity (optional, NULL ok)
 * router_bias may be NULL (no bias). Required: x, w_router, topk_idx, topk_w,
 * aux_loss, drop_mask, workspace; with T = 0 the [T,...] pointers may be NULL.
 */
int moe_route(const moe_cfg* cfg, const void* x, const void* w_router,
              const float* router_bias, int32_t* topk_idx, float* topk_w,
              float* aux_loss, uint8_t* drop_mask, int32_t* expert_counts,
              int32_t* kept_counts, void* workspace, size_t workspace_bytes,
              void* stream);

/*
 * The whole layer forward: routing as in moe_route, then each kept slot runs its
 * expert's SwiGLU FFN W2 (silu(W1 x) * (W3 x)) (2kiu.com/news/2885792 section 2.2)
 * and out[t] = sum over kept slots of topk_w[t,s] * expert output
 * (cf-1.com/news/5914943 section 2.1). Dropped slots contribute 0 and the kept
 * slots keep their weights; the residual is NOT added (the caller adds x), so a
 * token whose every slot was dropped gets out = 0. Required: x, w_router, w1, w3,
 * w2, out, workspace (x and out may be NULL when T = 0). Optional (NULL ok):
 * router_bias and the routing outputs.
 */
int moe_forward(const moe_cfg* cfg, const void* x, const void* w_router,
                const float* router_bias, const void* w1, const void* w3,
                const void* w2, void* out, int32_t* topk_idx, float* topk_w,
                float* aux_loss, uint8_t* drop_mask, int32_t* expert_counts,
                int32_t* kept_counts, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * moe_forward with stage timing: `stage_events` holds MOE_NUM_STAGES+1 cudaEvent_t
 * handles created by the caller; event i is recorded on `stream` before stage i and
 * event MOE_NUM_STAGES after the last stage. Stages: 0 router logits, 1 routing
 * decisions (softmax, top-k, gate weights, aux loss, capacity ranks and offsets),
 * 2 dispatch (permute), 3 expert GEMM1 + SwiGLU, 4 expert GEMM2, 5 gated combine.
 * bf16 layers with T > 3968 compute the router logits inside the routing-decision
 * kernel, so their stage 0 is empty and stage 1 holds both. NULL stage_events behaves
 * as moe_forward.
 */
int moe_forward_timed(const moe_cfg* cfg, const void* x, const void* w_router,
                      const float* router_bias, const void* w1, const void* w3,
                      const void* w2, void* out, int32_t* topk_idx, float* topk_w,
                      float* aux_loss, uint8_t* drop_mask, int32_t* expert_counts,
                      int32_t* kept_counts, void* workspace, size_t workspace_bytes,
                      void* stream, void* const* stage_events);

/*
 * Synchronise `stream`, read and clear the workspace status word. Returns MOE_OK,
 * MOE_EDEVICE (a kernel reported a failure; *bits, if not NULL, gets the word) or
 * MOE_ECUDA. Bits: 1 a bounded wait gave up, 2 an index out of range, 4 a kernel's
 * shared-memory layout did not fit its allocation (the kernel did no work).
 */
int moe_get_status(void* workspace, size_t workspace_bytes, void* stream,
                   uint32_t* bits);

/*
 * Routing without a caller-provided workspace, for callers that cannot allocate
 * device memory: plugin hosts and serving runtimes that plan every device buffer
 * up front and forbid a kernel library from calling cudaMalloc (an allocation can
 * synchronise the device, and fails once the runtime has reserved the memory).
 * The pages have no counterpart of this call; it computes exactly what moe_route
 * computes, with the same arguments minus the workspace.
 *
 * Its scratch is a static device array of MOE_STATIC_SCRATCH_BYTES inside this
 * library, which every GPU that loads the library holds until the process exits.
 * The call allocates nothing. It returns MOE_EUNSUPPORTED when the layer's routing
 * scratch does not fit that array (roughly: ksplit*T*N*4 partial logits plus about
 * 16*T*k bytes; every named workload here fits). The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress) with that device current and
 * keeps it for the life of the process; do not use this call on a device after
 * cudaDeviceReset() on it (the kept address would be stale). All calls share the
 * array and it keeps the last call's contents: calls that overlap on the GPU (other
 * streams, other threads) race and must be serialised by the caller. Each call clears
 * the array's status word before its kernels run; moe_get_status_static() reads what
 * they reported.
 */
#define MOE_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

int moe_route_static(const moe_cfg* cfg, const void* x, const void* w_router,
                     const float* router_bias, int32_t* topk_idx, float* topk_w,
                     float* aux_loss, uint8_t* drop_mask, int32_t* expert_counts,
                     int32_t* kept_counts, void* stream);

/*
 * moe_get_status for moe_route_static: synchronise `stream`, then read and clear the
 * status word of the static scratch array on the current device. Returns MOE_OK,
 * MOE_EDEVICE (*bits, if not NULL, gets the word; bits as in moe_get_status),
 * MOE_ECUDA or MOE_ENODEVICE. Allocates nothing.
 */
int moe_get_status_static(void* stream, uint32_t* bits);

/*
 * ---------------------------------------------------------------------------
 * Layer options: the variants the pages describe beyond the base layer. The
 * *_ex calls take a moe_options pointer; NULL means the base layer, exactly as
 * moe_workspace_size / moe_route / moe_forward_timed compute it.
 * ---------------------------------------------------------------------------
 */

/* Expert FFN. SWIGLU: W2 (silu(W1 x) * (W3 x)) (2kiu.com/news/2885792 section 2.2).
 * GELU: the two-layer expert W2 gelu(W1 x) with the exact (erf) GELU
 * (devpress.csdn.net MoE page section 4.1); w3 is not read and may be NULL. */
typedef enum { MOE_ACT_SWIGLU = 0, MOE_ACT_GELU = 1 } moe_activation;

/* Most shared experts one layer may have. */
#define MOE_MAX_SHARED 8

typedef struct {
  /* Shared experts (hotelren.com/news/5904824 section 3.3): always-on experts that
   * every valid token runs with weight 1, beside its k routed ones. They take no
   * capacity and stay out of the router, the counts and the losses. Their weights
   * follow the routed experts' in w1, w3, w2, which then hold N + n_shared experts
   * ([N+n_shared, F, H] and [N+n_shared, H, F]). 0 <= n_shared <= MOE_MAX_SHARED. */
  int32_t n_shared;
  /* moe_activation of every expert, routed and shared. */
  int32_t activation;
  /* [T] device bytes, 1 = real token, 0 = padding; NULL = every token is real.
   * Capacity counts only the real tokens (devpress.csdn.net MoE page section 5.2):
   * the layer treats the real tokens as its whole batch (T_valid of them, in token
   * order) for the counts, C = ceil(CF*T_valid*k/N), the ranks and every loss. A
   * padding token gets topk_idx -1, topk_w 0, every slot dropped, and out = 0. */
  const uint8_t* valid_mask;
  /* [1] device float32 or NULL: KL(uniform || f) with f_e = counts_e/(T_valid*k)
   * (hotelren.com/news/3071227 section 4.2 takes the KL divergence of the expert
   * load to the uniform target); +inf when some expert receives no slot; 0 when
   * T_valid = 0. */
  float* aux_kl;
  /* [1] device float32 or NULL: the unbiased variance (the square of the sample
   * standard deviation) of all T_valid*N router probabilities
   * (2kiu.com/news/2885792 section 5.1 penalises std(router_probs)^2); 0 when
   * T_valid = 0, NaN when T_valid*N = 1. */
  float* aux_std2;
  /* Nonzero: overflow rerouting instead of dropping. One round after the capacity
   * step (cf-1.com/news/5914943 section 2.3 note moves overflow tokens to idle
   * experts; hotelren.com/news/5904824 section 3.4 and 2kiu.com/news/2885792
   * section 2.2 send them to the next-best expert; hotelren.com/news/3071227
   * section 4.2 masks the overloaded experts and takes the best remaining one):
   * an expert has room when fewer than C slots chose it; a token's dropped slots,
   * in slot order, propose its best, second best, ... experts with room that it did
   * not select (logit descending, ties to the lower id); each expert accepts
   * proposals in token order up to C - count; the rest stay dropped. A moved slot
   * keeps its gate weight, topk_idx reports its new expert, drop_mask its final
   * state and kept_counts the final rows per expert; expert_counts and the losses
   * stay those of the original routing. No effect without a capacity limit. */
  int32_t reroute;
} moe_options;

/* Workspace bytes for cfg with opts (NULL opts: moe_workspace_size); 0 when cfg
 * or opts is invalid or unsupported. Pure host function. */
size_t moe_workspace_size_ex(const moe_cfg* cfg, const moe_options* opts);

/* moe_route with options: valid_mask, aux_kl, aux_std2 and reroute apply; n_shared and
 * activation do not change the routing (they only size the workspace). The
 * workspace must hold moe_workspace_size_ex(cfg, opts) bytes. Returns MOE_EINVAL
 * for an out-of-range n_shared or activation. */
int moe_route_ex(const moe_cfg* cfg, const moe_options* opts, const void* x,
                 const void* w_router, const float* router_bias, int32_t* topk_idx,
                 float* topk_w, float* aux_loss, uint8_t* drop_mask,
                 int32_t* expert_counts, int32_t* kept_counts, void* workspace,
                 size_t workspace_bytes, void* stream);

/* moe_forward_timed with options (stage_events may be NULL; stage 3 is GEMM1 with
 * the chosen activation). out[t] = the routed sum as in moe_forward plus the sum of
 * the n_shared shared experts' outputs; padding tokens get 0. w3 may be NULL with
 * MOE_ACT_GELU. The workspace must hold moe_workspace_size_ex(cfg, opts) bytes. */
int moe_forward_ex(const moe_cfg* cfg, const moe_options* opts, const void* x,
                   const void* w_router, const float* router_bias, const void* w1,
                   const void* w3, const void* w2, void* out, int32_t* topk_idx,
                   float* topk_w, float* aux_loss, uint8_t* drop_mask,
                   int32_t* expert_counts, int32_t* kept_counts, void* workspace,
                   size_t workspace_bytes, void* stream, void* const* stage_events);

/*
 * How moe_forward / moe_forward_ex runs a layer: the plan the host derives from cfg
 * and opts alone (no CUDA call, no device needed). It is the plan those calls use,
 * so a caller can report or test it. The expert GEMMs' tile shape depends on whether
 * a router bias will be passed (has_bias, 0 or 1).
 */
typedef struct {
  int32_t fused_routing;   /* 1: the router GEMM and the routing decisions run as one
                              kernel (bf16 with at least 32 tiles of 128 tokens) */
  int32_t routing_block;   /* tokens per routing block (the unit of the per-block
                              counts that dispatch reads) */
  int32_t router_ksplit;   /* slices of H the router GEMM splits into (1 when fused) */
  int32_t gemm1_tile_rows; /* rows per GEMM1 work item: 256 on CTA pairs, else 128 */
  int32_t gemm2_tile_rows; /* the same for GEMM2 */
  int32_t launches;        /* kernel launches of one forward with T > 0 (T = 0: none) */
  int64_t capacity;        /* C without a valid-token mask; -1 for no limit */
  int64_t workspace_bytes; /* moe_workspace_size_ex(cfg, opts) */
  int32_t routing_threads; /* threads per block of the routing-decision kernel */
  int32_t routing_warp_finish; /* 1: the last routing block's per-expert scan, capacity,
                              loss and expert layout run in one warp, 0: in the block */
} moe_plan;

/* Fill *plan for cfg and opts (NULL opts: the base layer). Returns MOE_OK,
 * MOE_EINVAL (NULL cfg or plan, invalid cfg or options) or MOE_EUNSUPPORTED. */
int moe_describe(const moe_cfg* cfg, const moe_options* opts, int has_bias, moe_plan* plan);

/* Static description of a status code. */
const char* moe_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
