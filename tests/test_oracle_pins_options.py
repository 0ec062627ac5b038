"""Pins of the oracle's optional features (shared experts, the GELU expert, the
valid-token mask, the KL and variance balance losses) to library routines, closed
forms and invariants that do not come from the oracle itself."""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch
import torch.nn.functional as Fn

import oracle as orc
from mixture_experts_layer_102_b300 import configs, inputs


def _t(a):
    return torch.from_numpy(np.asarray(a, np.float64))


def _torch_swiglu(x, w1, w3, w2):
    return Fn.linear(Fn.silu(Fn.linear(_t(x), _t(w1))) * Fn.linear(_t(x), _t(w3)), _t(w2)).numpy()


def _torch_gelu_ffn(x, w1, w2):
    return Fn.linear(Fn.gelu(Fn.linear(_t(x), _t(w1))), _t(w2)).numpy()


# ------------------------------------------------------------- balance losses

def test_kl_is_zero_for_uniform_routing():
    N, k = 8, 2
    v = np.linspace(-1.0, 2.0, N) ** 3
    x = np.stack([np.roll(v, t) for t in range(4 * N)])
    r = orc.route(x, np.eye(N), None, k, None)
    assert abs(r["aux_kl"]) < 1e-15


def test_kl_matches_scipy_entropy():
    rng = np.random.default_rng(21)
    for _ in range(20):
        N, k = int(rng.integers(2, 12)), 1
        x = rng.standard_normal((400, 16))
        r = orc.route(x, rng.standard_normal((16, N)), None, k, None)
        f = r["expert_counts"] / r["expert_counts"].sum()
        if (f == 0).any():
            assert r["aux_kl"] == math.inf
        else:
            assert abs(r["aux_kl"] - scipy.stats.entropy(np.full(N, 1.0 / N), f)) < 1e-12


def test_kl_two_expert_closed_form():
    # k=1, N=2, three tokens to expert 0 and one to expert 1: f = (3/4, 1/4),
    # KL(uniform || f) = 1/2 log(2/3) + 1/2 log(2) = 1/2 log(4/3)
    x = np.array([[2.0, 0.0], [3.0, 1.0], [1.0, 0.5], [0.0, 2.0]])
    r = orc.route(x, np.eye(2), None, 1, None)
    assert r["expert_counts"].tolist() == [3, 1]
    assert abs(r["aux_kl"] - 0.5 * math.log(4.0 / 3.0)) < 1e-15


def test_probability_variance_matches_torch_std():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((300, 32))
    r = orc.route(x, rng.standard_normal((32, 16)), None, 2, None)
    ref = torch.std(_t(r["probs"])).item() ** 2
    assert abs(r["aux_std2"] - ref) < 1e-15


def test_probability_variance_closed_forms():
    r = orc.route(np.random.default_rng(0).standard_normal((9, 8)), np.zeros((8, 5)), None, 2,
                  None)
    assert abs(r["aux_std2"]) < 1e-30                  # every P = 1/N (up to rounding)
    # two tokens, two experts: entries {p, 1-p, q, 1-q} around the mean 1/2
    x = np.array([[0.3, 0.0], [0.0, 1.1]])
    r = orc.route(x, np.eye(2), None, 1, None)
    p, q = scipy.special.expit(0.3), scipy.special.expit(-1.1)
    expect = (2 * (p - 0.5) ** 2 + 2 * (q - 0.5) ** 2) / 3.0
    assert abs(r["aux_std2"] - expect) < 1e-15


# ---------------------------------------------------------------- GELU expert

def test_gelu_against_torch_and_the_normal_cdf():
    z = np.linspace(-12.0, 12.0, 481)
    scale = np.maximum(np.abs(z), 1.0)
    assert (np.abs(orc.gelu(z) - Fn.gelu(_t(z)).numpy()) / scale).max() < 1e-15
    assert (np.abs(orc.gelu(z) - z * scipy.special.ndtr(z)) / scale).max() < 1e-15
    assert orc.gelu(np.array([0.0]))[0] == 0.0


def test_gelu_expert_orientation_and_library():
    H, F = 6, 4
    a, b, d = 2, 5, 1
    w1 = np.zeros((F, H)); w1[a, b] = 1.0
    w2 = np.zeros((H, F)); w2[d, a] = 1.0
    x = np.random.default_rng(23).standard_normal((3, H))
    expect = np.zeros((3, H))
    expect[:, d] = x[:, b] * scipy.special.ndtr(x[:, b])
    assert np.abs(orc.gelu_expert(x, w1, w2) - expect).max() < 1e-15
    rng = np.random.default_rng(24)
    w1, w2 = rng.standard_normal((40, 24)) / 5, rng.standard_normal((24, 40)) / 6
    xx = rng.standard_normal((10, 24))
    ref = _torch_gelu_ffn(xx, w1, w2)
    assert np.abs(orc.gelu_expert(xx, w1, w2) - ref).max() < 1e-12 * np.abs(ref).max()


def test_gelu_layer_k_equals_n_is_the_dense_mixture():
    cfg = configs.TINY_F32.with_(k=8)
    inp = inputs.make_inputs(cfg)
    x, wr = inp.x.astype(np.float64), inp.w_router.astype(np.float64)
    res = orc.moe_forward(x, wr, None, inp.w1, None, inp.w2, 8, None, activation="gelu")
    p = scipy.special.softmax(x @ wr, axis=1)
    dense = sum(p[:, e:e + 1] * _torch_gelu_ffn(x, inp.w1[e], inp.w2[e]) for e in range(8))
    assert np.abs(res.out - dense).max() < 1e-12 * np.abs(dense).max()


# -------------------------------------------------------------- shared experts

def _with_shared(cfg, n_shared, zero_routed_w2=False):
    big = cfg.with_(N=cfg.N + n_shared)
    inp = inputs.make_inputs(big)
    wr = inp.w_router[:, :cfg.N].copy()
    w2 = inp.w2.copy()
    if zero_routed_w2:
        w2[:cfg.N] = 0.0
    return inp, wr, w2


def test_shared_experts_alone_are_dense_ffns():
    cfg = configs.TINY_F32
    inp, wr, w2 = _with_shared(cfg, 2, zero_routed_w2=True)
    res = orc.moe_forward(inp.x, wr, None, inp.w1, inp.w3, w2, cfg.k, None, n_shared=2)
    ref = sum(_torch_swiglu(inp.x, inp.w1[cfg.N + j], inp.w3[cfg.N + j], w2[cfg.N + j])
              for j in range(2))
    assert np.abs(res.out - ref).max() < 1e-12 * np.abs(ref).max()


def test_shared_expert_adds_to_the_routed_output():
    cfg = configs.TINY_F32.with_(capacity_factor=0.8)
    inp, wr, w2 = _with_shared(cfg, 1)
    routed = orc.moe_forward(inp.x, wr, None, inp.w1[:cfg.N], inp.w3[:cfg.N], w2[:cfg.N],
                             cfg.k, 0.8)
    both = orc.moe_forward(inp.x, wr, None, inp.w1, inp.w3, w2, cfg.k, 0.8, n_shared=1)
    shared = _torch_swiglu(inp.x, inp.w1[cfg.N], inp.w3[cfg.N], w2[cfg.N])
    assert np.abs(both.out - (routed.out + shared)).max() < 1e-12 * np.abs(both.out).max()
    assert both.aux_loss == routed.aux_loss and (both.drop_mask == routed.drop_mask).all()


# ------------------------------------------------------------ valid-token mask

def test_all_valid_mask_changes_nothing():
    cfg = configs.TINY_F32.with_(capacity_factor=0.7)
    inp = inputs.make_inputs(cfg)
    a = orc.moe_forward(inp.x, inp.w_router, None, inp.w1, inp.w3, inp.w2, 2, 0.7)
    b = orc.moe_forward(inp.x, inp.w_router, None, inp.w1, inp.w3, inp.w2, 2, 0.7,
                        valid_mask=np.ones(cfg.T, np.uint8))
    assert (a.out == b.out).all() and (a.drop_mask == b.drop_mask).all()
    assert a.aux_loss == b.aux_loss and a.capacity == b.capacity


def test_capacity_counts_only_valid_tokens():
    # 12 tokens, 6 of them padding: C = ceil(1.0 * 6 * 2 / 4) = 3, not ceil(12*2/4) = 6
    rng = np.random.default_rng(25)
    x = rng.standard_normal((12, 8))
    mask = np.array([1, 0, 1, 1, 0, 0, 1, 0, 1, 0, 1, 0], np.uint8)
    r = orc.route(x, rng.standard_normal((8, 4)), None, 2, 1.0, valid_mask=mask)
    assert r["capacity"] == 3
    pad = mask == 0
    assert (r["topk_idx"][pad] == -1).all() and (r["topk_w"][pad] == 0).all()
    assert (r["drop_mask"][pad] == 1).all()
    assert r["expert_counts"].sum() == 6 * 2


def test_padding_tokens_get_zero_even_with_shared_experts():
    cfg = configs.TINY_F32.with_(capacity_factor=1.0)
    inp, wr, w2 = _with_shared(cfg, 1)
    mask = (np.arange(cfg.T) % 3 != 1).astype(np.uint8)
    res = orc.moe_forward(inp.x, wr, None, inp.w1, inp.w3, w2, cfg.k, 1.0, n_shared=1,
                          valid_mask=mask)
    assert (res.out[mask == 0] == 0).all()
    assert np.abs(res.out[mask == 1]).max() > 0


# --------------------------------------------------------- overflow rerouting

def _route_logits(logits, k, cf, **kw):
    """Route with the logits given directly: identity router over H = N."""
    logits = np.asarray(logits, np.float64)
    return orc.route(logits, np.eye(logits.shape[1]), None, k, cf, **kw)


def test_reroute_hand_example_k1():
    # C = ceil(0.75 * 5 * 1 / 4) = 1. Tokens 0, 1, 2, 4 pick expert 0, token 3 expert 3.
    # Experts 1 and 2 have room: token 1 moves to 2 (its better one), token 2 to 1,
    # token 4 also wants 1 but it is full by then, so it stays dropped.
    L = [[3, 2, 1, 0], [3, 0, 2, 1], [3, 1, 0, 2], [0, 1, 2, 3], [3, 2, 1.5, 0]]
    r = _route_logits(L, 1, 0.75, reroute=True)
    assert r["capacity"] == 1
    assert r["topk_idx"][:, 0].tolist() == [0, 2, 1, 3, 0]
    assert r["drop_mask"][:, 0].tolist() == [0, 0, 0, 0, 1]
    assert r["rerouted"][:, 0].tolist() == [0, 1, 1, 0, 0]
    assert r["kept_counts"].tolist() == [1, 1, 1, 1]
    assert r["expert_counts"].tolist() == [4, 0, 0, 1]      # before capacity, unchanged


def test_reroute_excludes_the_tokens_own_experts():
    # C = ceil(1.0 * 3 * 2 / 5) = 2; expert 0 overflows by one (token 2). Token 2's own
    # expert 4 has room and the larger logit, but a token visits an expert at most
    # once: it moves to expert 1.
    L = [[4, 3, 0, 0, 0], [4, 0, 3, 2, 1], [4, 2.5, 0, 1, 3]]
    r = _route_logits(L, 2, 1.0, reroute=True)
    assert r["capacity"] == 2
    assert r["topk_idx"].tolist() == [[0, 1], [0, 2], [1, 4]]
    assert r["drop_mask"].sum() == 0 and r["rerouted"].tolist() == [[0, 0], [0, 0], [1, 0]]
    assert r["kept_counts"].tolist() == [2, 2, 1, 0, 1]


def test_reroute_slots_take_candidates_in_slot_order():
    # C = ceil(1.0 * 2 * 2 / 6) = 1: token 1 loses both slots; they take its best and
    # second best experts with room (3, then 4).
    L = [[5, 4, 0, 0, 0, 0], [5, 4, 1, 3, 2, 0]]
    r = _route_logits(L, 2, 1.0, reroute=True)
    assert r["topk_idx"].tolist() == [[0, 1], [3, 4]]
    assert r["drop_mask"].sum() == 0


def test_reroute_keeps_gate_weights_and_base_when_nothing_overflows():
    rng = np.random.default_rng(26)
    x, wr = rng.standard_normal((200, 16)), rng.standard_normal((16, 8))
    a = orc.route(x, wr, None, 2, 4.0)
    b = orc.route(x, wr, None, 2, 4.0, reroute=True)         # C = 200: no drops
    assert a["drop_mask"].sum() == 0 and (a["topk_idx"] == b["topk_idx"]).all()
    c = orc.route(x, wr, None, 2, 0.5, reroute=True)
    d = orc.route(x, wr, None, 2, 0.5)
    assert (c["topk_w"] == d["topk_w"]).all() and c["aux_loss"] == d["aux_loss"]
    # k = N: no expert left to move to
    e = orc.route(x, wr, None, 8, 0.5, reroute=True)
    f = orc.route(x, wr, None, 8, 0.5)
    assert (e["topk_idx"] == f["topk_idx"]).all() and (e["drop_mask"] == f["drop_mask"]).all()


@pytest.mark.parametrize("cf", [0.3, 0.8, 1.0])
def test_reroute_invariants(cf):
    cfg = configs.TINY_F32.with_(T=600, N=16, k=2, capacity_factor=cf, zipf_bias=True)
    inp = inputs.make_inputs(cfg, with_experts=False)
    base = orc.route(inp.x, inp.w_router, inp.router_bias, 2, cf)
    r = orc.route(inp.x, inp.w_router, inp.router_bias, 2, cf, reroute=True)
    C, N = r["capacity"], 16
    idx, drop, rer = r["topk_idx"], r["drop_mask"], r["rerouted"]
    final_counts = np.bincount(idx[drop == 0], minlength=N)
    assert (final_counts == r["kept_counts"]).all() and (final_counts <= C).all()
    assert r["drop_mask"].sum() <= base["drop_mask"].sum()
    assert ((rer == 1) <= (base["drop_mask"] == 1)).all()             # only dropped slots move
    assert (idx[base["drop_mask"] == 0] == base["topk_idx"][base["drop_mask"] == 0]).all()
    for t in np.nonzero(rer.any(axis=1))[0]:
        assert len(set(idx[t].tolist())) == 2                          # still distinct
        for s in np.nonzero(rer[t])[0]:
            e = idx[t, s]
            assert e not in base["topk_idx"][t] and base["expert_counts"][e] < C
    # a slot that stays dropped was turned away: the expert it proposed (its token's
    # j-th best expert with room that the token did not select, j = the slot's place
    # among the token's dropped slots) ends up full; brute force over the experts
    room_left = C - final_counts
    logits = base["logits"]
    for t in np.nonzero(drop.any(axis=1))[0]:
        lost = [s for s in range(2) if base["drop_mask"][t, s]]
        allowed = sorted((e for e in range(N) if base["expert_counts"][e] < C
                          and e not in base["topk_idx"][t]),
                         key=lambda e: (-logits[t, e], e))
        for j, s in enumerate(lost):
            if drop[t, s] and j < len(allowed):
                assert room_left[allowed[j]] == 0, (t, s, allowed[j])
            elif not drop[t, s]:
                assert idx[t, s] == allowed[j]


# ------------------------------------------- near ties of the rerouting proposals

def _near(logits, idx, drop, counts, C):
    return orc.reroute_near_ties(np.asarray(logits, np.float64)[None, :],
                                 np.asarray([idx]), np.asarray([drop], np.uint8),
                                 np.asarray(counts), C).tolist()


def test_reroute_near_tie_listed_when_the_best_two_candidates_are_close():
    # one dropped slot (m = 1): its proposal is the best expert with room that the
    # token did not select; experts 3 and 2 (both with room) are 5e-5 apart, so the
    # proposal may flip between them
    L = [9, 8, 3.0, 3.00005, 1, 0]
    assert _near(L, [0, 1], [0, 1], [5, 5, 0, 0, 0, 0], 2) == [0]
    # 1e-3 apart: the proposal is decided
    L2 = [9, 8, 3.0, 3.001, 1, 0]
    assert _near(L2, [0, 1], [0, 1], [5, 5, 0, 0, 0, 0], 2) == []


def test_reroute_near_tie_looks_at_m_plus_one_candidates_only():
    # m = 1: the best candidate (expert 2) is far ahead; the close pair (4, 3) is the
    # second and third candidate, which cannot change the one proposal
    L = [9, 8, 5.0, 3.0, 3.00005, 0]
    assert _near(L, [0, 1], [0, 1], [5, 5, 0, 0, 0, 0], 2) == []
    # m = 2 (both slots dropped): the second proposal is between 4 and 3
    assert _near(L, [0, 1], [1, 1], [5, 5, 0, 0, 0, 0], 2) == [0]


def test_reroute_near_tie_skips_full_and_own_experts():
    L = [9, 8, 3.0, 3.00005, 1, 0]
    # expert 3 is full (count 2 = C): the candidates are 2, 4, 5, far apart
    assert _near(L, [0, 1], [0, 1], [5, 5, 0, 2, 0, 0], 2) == []
    # the token's own expert 1 sits next to candidate 2 but is not a candidate
    L3 = [9, 3.00005, 3.0, 1, 0.5, 0]
    assert _near(L3, [0, 1], [0, 1], [5, 0, 0, 0, 0, 0], 2) == []


def test_reroute_near_tie_empty_without_drops_or_capacity():
    L = [9, 8, 3.0, 3.00005, 1, 0]
    assert _near(L, [0, 1], [0, 0], [5, 5, 0, 0, 0, 0], 2) == []
    assert _near(L, [0, 1], [0, 1], [5, 5, 0, 0, 0, 0], None) == []


def _proposals(logits_t, idx_t, counts, C, m):
    """The m proposals of a token by brute force: every expert with room that the
    token did not select, ordered by (logit desc, id asc)."""
    cand = sorted((e for e in range(len(logits_t)) if counts[e] < C and e not in idx_t),
                  key=lambda e: (-logits_t[e], e))
    return cand[:m]


def test_reroute_near_ties_are_exactly_the_unstable_proposals():
    # On a Zipf-skewed batch whose logits are rounded to a 1e-4 grid (so that many
    # candidates tie or sit one grid step apart): a token that is NOT listed keeps its
    # proposals under every perturbation of its logits by less than half the margin,
    # and a listed one changes them when the closest pair among its first m+1
    # candidates moves apart in the other direction by about half the margin each.
    cfg = configs.TINY_F32.with_(T=400, N=12, k=2, capacity_factor=0.7, zipf_bias=True)
    inp = inputs.make_inputs(cfg, with_experts=False)
    base = orc.route(inp.x, inp.w_router, inp.router_bias, 2, 0.7)
    logits = np.round(base["logits"] * 1e4) / 1e4
    idx = orc.topk_select(logits, 2)
    counts = orc.expert_counts(idx, 12)
    C = base["capacity"]
    _, drop, _ = orc.capacity_assign(idx, 12, C)
    listed = set(orc.reroute_near_ties(logits, idx, drop, counts, C).tolist())
    rng = np.random.default_rng(3)
    n_listed = n_stable = 0
    for t in np.nonzero(drop.any(axis=1))[0]:
        m = int(drop[t].sum())
        prop = _proposals(logits[t], idx[t].tolist(), counts, C, m)
        if t in listed:
            n_listed += 1
            cand = _proposals(logits[t], idx[t].tolist(), counts, C, m + 1)
            v = logits[t][cand]
            j = int(np.argmin(v[:-1] - v[1:]))
            delta = 0.5 * (v[j] - v[j + 1]) + 1e-7   # < half the margin plus 1e-7
            assert delta < 0.5e-4 + 1e-7
            swapped = logits[t].copy()
            swapped[cand[j]] -= delta
            swapped[cand[j + 1]] += delta
            assert _proposals(swapped, idx[t].tolist(), counts, C, m) != prop
        else:
            n_stable += 1
            for _ in range(20):
                noisy = logits[t] + rng.uniform(-0.49e-4, 0.49e-4, size=12)
                assert _proposals(noisy, idx[t].tolist(), counts, C, m) == prop
    assert n_listed > 0 and n_stable > 0
