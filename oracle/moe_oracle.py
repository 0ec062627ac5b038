"""Plain CPU fp64 oracle of the forward pass of one top-k routed MoE FFN layer.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's CPU
baseline leg import this module. The product path (the CUDA library and its Python
binding) never calls it, and it shares no code with that path: it receives plain
arrays (the same bf16-rounded values the GPU gets, as float32) and widens them to
float64 itself.

What it computes, step by step, in the pages' order:

1. router logits  l = x @ W_r (+ b)           -- a small linear layer [hidden, N]
   (cf-1.com/news/5914943 section 2.1; 2kiu.com/news/2885792 section 3.1)
2. full router softmax P = softmax(l)          -- used only by the aux loss
   (cf-1.com/news/5914943 section 2.3; devpress.csdn.net MoE page section 4.1)
3. top-k over the logits, ties to the lower expert id, then a softmax over the k
   selected logits (cf-1.com/news/5914943 section 2.1; hotelren.com/news/3071227
   section 4.1; stable tie order: 2kiu.com/news/2885792 section 5.3)
4. aux = N * sum_e f_e * P_e with f_e the fraction of routing slots sent to e and P_e
   the mean router probability of e (cf-1.com/news/5914943 section 2.3)
5. per-expert capacity C = ceil(CF*T*k/N); each expert keeps the first C routed tokens
   in token order and drops the rest to the residual (cf-1.com/news/5914943 section
   2.3 note; 2kiu.com/news/2885792 sections 2.2 and 3.1)
6. each kept slot runs the expert's SwiGLU FFN  W2 (silu(W1 x) * (W3 x))
   (2kiu.com/news/2885792 section 2.2 names SwiGLU as the expert FFN)
7. combine y[t] = sum over kept slots of w[t,s] * expert output
   (cf-1.com/news/5914943 section 2.1; hotelren.com/news/5904824 section 3.1)

Readings where the pages are open (each also listed in the design notes):
* f_e = counts_e / (T*k), so sum_e f_e = 1 and a balanced router gives aux = 1 (the
  pages say the ideal value is about 1); counts are taken BEFORE capacity.
* C = ceil(CF*T*k/N) evaluated in IEEE double from the float32 value of CF.
  capacity_factor None (or <= 0) means no limit.
* a dropped slot contributes 0 and the kept slots keep their original gate weights
  (no renormalisation); the layer returns only the MoE branch, the caller adds the
  residual, so a token with every slot dropped gets exactly 0.
* T = 0 gives aux = 0 (empty sums).

Options beyond the base layer (the pages' further variants):
* shared experts (hotelren.com/news/5904824 section 3.3): ``n_shared`` always-on experts
  whose weights follow the routed ones; every valid token adds their outputs with
  weight 1; they take no capacity and stay out of the router and the aux losses.
* the two-layer GELU expert W2 gelu(W1 x) (devpress.csdn.net MoE page section 4.1),
  exact (erf) GELU.
* a valid-token mask (devpress.csdn.net MoE page section 5.2: capacity counts only
  non-padding tokens). Reading: padding tokens are routed as if they were not in the
  batch at all -- everything (counts, capacity with T_valid, ranks, aux losses) is the
  layer on the valid tokens alone; padding tokens get no expert (index -1, weight 0,
  dropped) and output 0.
* overflow rerouting instead of dropping (cf-1.com/news/5914943 section 2.3 note
  moves overflow tokens to other, idle experts; hotelren.com/news/5904824 section 3.4
  and 2kiu.com/news/2885792 section 2.2 send them to the next-best expert; the
  capacity-aware routing of hotelren.com/news/3071227 section 4.2 masks the
  overloaded experts' logits and takes the best remaining one). Reading: one round.
  After the capacity step, the experts a token may move to are those that still
  have room (count < C) and that the token did not select; its dropped slots, in
  slot order, propose the best, second best, ... of them by logit (ties to the lower
  id), so a token still visits an expert at most once. Each expert accepts the
  proposals in token order (t, then slot) up to its remaining room C - count; the
  other slots stay dropped. A rerouted slot keeps its gate weight; its topk_idx
  becomes the new expert. Counts before capacity and the losses are those of the
  original routing.
* two more balance losses: KL(uniform || f) with f_e = counts_e / (T*k)
  (hotelren.com/news/3071227 section 4.2 takes the KL divergence of the expert load
  to the uniform target; its load is normalised by the mask size, here by T*k so that
  f is a distribution), and the unbiased variance of all router probabilities
  (2kiu.com/news/2885792 section 5.1: lambda * std(router_probs)**2, without lambda).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

NEAR_TIE_MARGIN = 1e-4


def capacity(T: int, k: int, N: int, capacity_factor: Optional[float]) -> Optional[int]:
    """Per-expert capacity C = ceil(CF*T*k/N), or None for no limit.

    CF is the layer's float32 value; the product is evaluated left to right in
    double: ((CF*T)*k)/N.
    """
    if capacity_factor is None or capacity_factor <= 0:
        return None
    cf = float(np.float32(capacity_factor))
    return int(math.ceil(cf * T * k / N))


def capacity_page_example_variant(num_tokens: int, num_experts: int, cf: float) -> int:
    """The worked capacity example's own formula: floor(CF * tokens / experts), with
    no top-k factor (hotelren.com/news/3071227 section 2.2). Not used by the layer;
    it only reproduces the page's printed numbers."""
    return int(math.floor(cf * num_tokens / num_experts))


def router_logits(x: np.ndarray, w_router: np.ndarray,
                  bias: Optional[np.ndarray] = None) -> np.ndarray:
    """l[t,e] = sum_h x[t,h] * W_r[h,e] (+ b[e]), in float64."""
    l = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64)
    if bias is not None:
        l = l + np.asarray(bias, np.float64)[None, :]
    return l


def full_softmax(logits: np.ndarray) -> np.ndarray:
    """Row-wise softmax over all N experts (max subtracted first)."""
    m = logits.max(axis=1, keepdims=True) if logits.shape[0] else 0.0
    e = np.exp(logits - m)
    return e / e.sum(axis=1, keepdims=True)


def topk_select(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, ordered by logit descending; equal
    logits are ordered by ascending expert id (the stable tie rule)."""
    T, N = logits.shape
    ids = np.broadcast_to(np.arange(N), (T, N))
    # np.lexsort sorts by the LAST key first: primary -logit, secondary id.
    order = np.lexsort((ids, -logits), axis=-1)
    return order[:, :k].astype(np.int64)


def gate_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Softmax over the k selected logits of each token."""
    sel = np.take_along_axis(logits, idx, axis=1)
    e = np.exp(sel - sel[:, :1]) if sel.shape[0] else sel
    return e / e.sum(axis=1, keepdims=True)


def expert_counts(idx: np.ndarray, N: int) -> np.ndarray:
    """Number of routing slots sent to each expert (before capacity)."""
    return np.bincount(idx.ravel(), minlength=N).astype(np.int64)


def aux_loss(probs: np.ndarray, idx: np.ndarray, N: int, k: int) -> float:
    """aux = N * sum_e f_e * P_e, f_e = counts_e/(T*k), P_e = mean_t P[t,e]."""
    T = idx.shape[0]
    if T == 0:
        return 0.0
    f = expert_counts(idx, N) / float(T * k)
    P = probs.mean(axis=0)
    return float(N * np.sum(f * P))


def aux_kl_uniform(idx: np.ndarray, N: int, k: int) -> float:
    """KL(uniform || f) = sum_e (1/N) log((1/N) / f_e), f_e = counts_e/(T*k); +inf
    when an expert receives no slot, 0 for an empty batch."""
    T = idx.shape[0]
    if T == 0:
        return 0.0
    f = expert_counts(idx, N) / float(T * k)
    with np.errstate(divide="ignore"):
        return float(np.sum((1.0 / N) * (np.log(1.0 / N) - np.log(f))))


def aux_prob_variance(probs: np.ndarray) -> float:
    """Unbiased variance over all entries of the router probabilities (torch.std's
    default correction), squared std; 0 for an empty batch."""
    if probs.size == 0:
        return 0.0
    if probs.size == 1:
        return float("nan")
    return float(np.var(probs, ddof=1))


def capacity_assign(idx: np.ndarray, N: int, C: Optional[int]):
    """Walk the slots in token order (t ascending, then slot s) and give each the
    number of earlier slots that chose the same expert. A slot is dropped when that
    rank reaches C. Returns (rank[T,k], drop_mask[T,k] uint8, kept_counts[N])."""
    T, k = idx.shape
    rank = np.zeros((T, k), dtype=np.int64)
    seen = [0] * N
    for t in range(T):
        for s in range(k):
            e = int(idx[t, s])
            rank[t, s] = seen[e]
            seen[e] += 1
    if C is None:
        drop = np.zeros((T, k), dtype=np.uint8)
    else:
        drop = (rank >= C).astype(np.uint8)
    kept = np.zeros(N, dtype=np.int64)
    np.add.at(kept, idx[drop == 0], 1)
    return rank, drop, kept


def _reroute_candidates(logits_t, idx_t, has_room):
    """Experts token t may move to, best first: room left, not selected by t; by
    logit descending, ties to the lower id."""
    allowed = has_room.copy()
    allowed[idx_t] = False
    cand = np.nonzero(allowed)[0]
    return cand[np.lexsort((cand, -logits_t[cand]))]


def reroute_overflow(logits: np.ndarray, idx: np.ndarray, drop: np.ndarray,
                     counts: np.ndarray, C: Optional[int]):
    """One round of capacity-aware rerouting of the dropped slots (the reading in the
    header). Returns (idx_final[T,k], drop_final[T,k], rerouted[T,k] uint8,
    accepted[N] rerouted slots taken by each expert)."""
    T, k = idx.shape
    N = logits.shape[1]
    idx_f = idx.copy()
    drop_f = drop.copy()
    rerouted = np.zeros((T, k), dtype=np.uint8)
    accepted = np.zeros(N, dtype=np.int64)
    if C is None:
        return idx_f, drop_f, rerouted, accepted
    room = np.maximum(C - counts, 0)
    has_room = counts < C
    for t in range(T):
        dropped = [s for s in range(k) if drop[t, s]]
        if not dropped:
            continue
        cand = _reroute_candidates(logits[t], idx[t], has_room)
        for j, s in enumerate(dropped):
            if j >= cand.size:
                break
            c = int(cand[j])
            if accepted[c] < room[c]:
                accepted[c] += 1
                idx_f[t, s] = c
                drop_f[t, s] = 0
                rerouted[t, s] = 1
    return idx_f, drop_f, rerouted, accepted


def reroute_near_ties(logits: np.ndarray, idx: np.ndarray, drop: np.ndarray,
                      counts: np.ndarray, C: Optional[int],
                      margin: float = NEAR_TIE_MARGIN) -> np.ndarray:
    """Tokens whose m dropped slots' proposals may flip: two of the m+1 best
    candidates have logits within ``margin``."""
    out = []
    if C is None:
        return np.zeros(0, dtype=np.int64)
    has_room = counts < C
    for t in np.nonzero(drop.any(axis=1))[0]:
        m = int(drop[t].sum())
        cand = _reroute_candidates(logits[t], idx[t], has_room)
        v = logits[t][cand[:m + 1]]
        if v.size >= 2 and (v[:-1] - v[1:] < margin).any():
            out.append(t)
    return np.asarray(out, dtype=np.int64)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_expert(x_rows: np.ndarray, w1_e: np.ndarray, w3_e: np.ndarray,
                  w2_e: np.ndarray) -> np.ndarray:
    """One expert: W2 (silu(W1 x) * (W3 x)), weights in [out, in] orientation."""
    xr = np.asarray(x_rows, np.float64)
    g = xr @ np.asarray(w1_e, np.float64).T
    u = xr @ np.asarray(w3_e, np.float64).T
    return (silu(g) * u) @ np.asarray(w2_e, np.float64).T


def gelu(z: np.ndarray) -> np.ndarray:
    """Exact GELU: z * Phi(z) = 0.5 z (1 + erf(z / sqrt(2)))."""
    from scipy.special import erf
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def gelu_expert(x_rows: np.ndarray, w1_e: np.ndarray, w2_e: np.ndarray) -> np.ndarray:
    """The two-layer expert: W2 gelu(W1 x)."""
    xr = np.asarray(x_rows, np.float64)
    return gelu(xr @ np.asarray(w1_e, np.float64).T) @ np.asarray(w2_e, np.float64).T


def expert_ffn(x_rows, w1_e, w3_e, w2_e, activation: str = "swiglu") -> np.ndarray:
    if activation == "gelu":
        return gelu_expert(x_rows, w1_e, w2_e)
    return swiglu_expert(x_rows, w1_e, w3_e, w2_e)


def near_tie_tokens(logits: np.ndarray, k: int, margin: float = NEAR_TIE_MARGIN):
    """(set_ties, order_ties): tokens whose k-th and (k+1)-th largest logits differ by
    less than ``margin`` (the selected SET may flip), and tokens where two
    consecutive selected logits do (only the slot ORDER may flip)."""
    T, N = logits.shape
    s = -np.sort(-logits, axis=1)
    if k < N:
        set_ties = np.nonzero(s[:, k - 1] - s[:, k] < margin)[0]
    else:
        set_ties = np.zeros(0, dtype=np.int64)
    if k > 1:
        order_ties = np.nonzero((s[:, :k - 1] - s[:, 1:k] < margin).any(axis=1))[0]
    else:
        order_ties = np.zeros(0, dtype=np.int64)
    return set_ties, order_ties


def active_fraction(idx: np.ndarray, N: int) -> float:
    """Mean fraction of the N experts whose FFN a token runs (distinct experts)."""
    if idx.shape[0] == 0:
        return 0.0
    return float(np.mean([len(set(row.tolist())) for row in idx]) / N)


@dataclass
class OracleResult:
    logits: np.ndarray          # [T,N] float64
    probs: np.ndarray           # [T,N] float64
    topk_idx: np.ndarray        # [T,k] int64
    topk_w: np.ndarray          # [T,k] float64
    aux_loss: float
    expert_counts: np.ndarray   # [N] before capacity
    capacity: Optional[int]
    rank: np.ndarray            # [T,k]
    drop_mask: np.ndarray       # [T,k] uint8, 1 = dropped
    kept_counts: np.ndarray     # [N]
    tokens: np.ndarray          # token ids whose output rows are in ``out``
    out: np.ndarray             # [len(tokens), H] float64
    near_tie_set: np.ndarray
    near_tie_order: np.ndarray
    aux_kl: float = 0.0
    aux_std2: float = 0.0
    rerouted: Optional[np.ndarray] = None    # [T,k] uint8, 1 = slot moved by rerouting
    reroute_ties: Optional[np.ndarray] = None


def route(x, w_router, bias, k: int, capacity_factor, valid_mask=None, reroute=False):
    """Steps 1-5 for every token. With ``valid_mask``, the valid tokens are routed as
    a batch of their own and the padding tokens get index -1, weight 0, dropped. With
    ``reroute``, dropped slots take one round of rerouting (``reroute_overflow``)."""
    if valid_mask is not None:
        return _route_masked(x, w_router, bias, k, capacity_factor,
                             np.asarray(valid_mask).astype(bool), reroute)
    T = x.shape[0]
    N = w_router.shape[1]
    logits = router_logits(x, w_router, bias)
    probs = full_softmax(logits)
    idx = topk_select(logits, k)
    w = gate_weights(logits, idx)
    aux = aux_loss(probs, idx, N, k)
    counts = expert_counts(idx, N)
    C = capacity(T, k, N, capacity_factor)
    rank, drop, kept = capacity_assign(idx, N, C)
    set_ties, order_ties = near_tie_tokens(logits, k)
    r = dict(logits=logits, probs=probs, topk_idx=idx, topk_w=w, aux_loss=aux,
             aux_kl=aux_kl_uniform(idx, N, k), aux_std2=aux_prob_variance(probs),
             expert_counts=counts, capacity=C, rank=rank, drop_mask=drop,
             kept_counts=kept, near_tie_set=set_ties, near_tie_order=order_ties,
             rerouted=np.zeros((T, k), dtype=np.uint8),
             reroute_ties=np.zeros(0, dtype=np.int64))
    if reroute:
        idx_f, drop_f, rer, acc = reroute_overflow(logits, idx, drop, counts, C)
        r.update(topk_idx=idx_f, drop_mask=drop_f, rerouted=rer, kept_counts=kept + acc,
                 reroute_ties=reroute_near_ties(logits, idx, drop, counts, C))
    return r


def _route_masked(x, w_router, bias, k, capacity_factor, valid, reroute=False):
    T = x.shape[0]
    v = np.nonzero(valid)[0]
    r = route(np.asarray(x)[v], w_router, bias, k, capacity_factor, reroute=reroute)
    full = dict(r)
    full["logits"] = router_logits(x, w_router, bias)
    full["probs"] = full_softmax(full["logits"])
    idx = np.full((T, k), -1, dtype=np.int64)
    idx[v] = r["topk_idx"]
    w = np.zeros((T, k))
    w[v] = r["topk_w"]
    rank = np.full((T, k), -1, dtype=np.int64)
    rank[v] = r["rank"]
    drop = np.ones((T, k), dtype=np.uint8)
    drop[v] = r["drop_mask"]
    rer = np.zeros((T, k), dtype=np.uint8)
    rer[v] = r["rerouted"]
    full.update(topk_idx=idx, topk_w=w, rank=rank, drop_mask=drop, rerouted=rer,
                near_tie_set=v[r["near_tie_set"]], near_tie_order=v[r["near_tie_order"]],
                reroute_ties=v[r["reroute_ties"]], valid_tokens=v)
    return full


def experts_combine(x, w1, w3, w2, idx, w, drop, tokens, n_shared: int = 0,
                    activation: str = "swiglu", valid_mask=None) -> np.ndarray:
    """Steps 6-7 for the given routing decisions: every kept slot (t, s) of the tokens
    in ``tokens`` runs expert idx[t,s]'s FFN on x[t], and row i of the result is the
    sum of those outputs weighted by w[t,s] (dropped slots add nothing), plus the
    outputs of the ``n_shared`` shared experts (experts N.. of w1/w3/w2, weight 1) for
    the valid tokens. N is the number of routed experts: w1 holds N + n_shared."""
    H = x.shape[1]
    N = w1.shape[0] - n_shared
    tokens = np.asarray(tokens, np.int64)
    out = np.zeros((len(tokens), H), dtype=np.float64)
    k = idx.shape[1]
    # Queue every kept slot of the requested tokens on its expert.
    queue = [([], []) for _ in range(N)]
    for i, t in enumerate(tokens):
        for s in range(k):
            if not drop[t, s]:
                queue[int(idx[t, s])][0].append(i)
                queue[int(idx[t, s])][1].append(s)
    for e in range(N):
        rows, slots = queue[e]
        if not rows:
            continue
        rows = np.asarray(rows)
        slots = np.asarray(slots)
        # A token visits an expert at most once, so ``rows`` has no repeats here.
        ye = expert_ffn(np.asarray(x[tokens[rows]], np.float64), w1[e],
                        None if w3 is None else w3[e], w2[e], activation)
        out[rows] += w[tokens[rows], slots][:, None] * ye
    if n_shared:
        live = np.arange(len(tokens))
        if valid_mask is not None:
            live = live[np.asarray(valid_mask).astype(bool)[tokens]]
        if len(live):
            xs = np.asarray(x[tokens[live]], np.float64)
            for j in range(n_shared):
                e = N + j
                out[live] += expert_ffn(xs, w1[e], None if w3 is None else w3[e], w2[e],
                                        activation)
    return out


def moe_forward(x, w_router, bias, w1, w3, w2, k: int, capacity_factor,
                token_sample: Optional[np.ndarray] = None, n_shared: int = 0,
                activation: str = "swiglu", valid_mask=None,
                reroute: bool = False) -> OracleResult:
    """The whole layer. Routing and capacity always cover every token (capacity
    depends on token order); the expert FFN and the combine are evaluated for the
    tokens in ``token_sample`` (all tokens when None). w1/w3/w2 hold the N routed
    experts followed by ``n_shared`` shared ones (w3 unused for GELU experts)."""
    T = x.shape[0]
    r = route(x, w_router, bias, k, capacity_factor, valid_mask, reroute)
    tokens = np.arange(T) if token_sample is None else np.asarray(token_sample, np.int64)
    out = experts_combine(x, w1, w3, w2, r["topk_idx"], r["topk_w"], r["drop_mask"], tokens,
                          n_shared, activation, valid_mask)
    r = {key: val for key, val in r.items() if key in OracleResult.__dataclass_fields__}
    return OracleResult(out=out, tokens=tokens, **r)
