"""Pins of the fp64 oracle to facts that do not come from the oracle itself:
values the pages print, closed forms of special cases, invariants, brute force on tiny
inputs and independent library routines (scipy, torch CPU float64).

Each pin is chosen so that a plausible mistake in the oracle fails it: a floor instead
of a ceil in the capacity, a missing top-k factor in f_e, counts taken after capacity,
a reversed tie rule, a softmax over all experts instead of the k selected, gate weights
renormalised after a drop, a transposed or swapped expert weight, a wrong silu sign.
"""
import itertools
import math
from pathlib import Path

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as Fn

import oracle as orc
from mixture_experts_layer_102_b300 import configs, inputs

GOLDEN = Path(__file__).parent / "golden"


def _kv(path):
    out = {}
    for line in path.read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            for tok in line.split():
                key, val = tok.split("=")
                out.setdefault(key, []).append(val)
    return out


def _torch_swiglu(x, w1, w3, w2):
    """Independent float64 SwiGLU through torch's own linear and silu."""
    xt = torch.from_numpy(np.asarray(x, np.float64))
    g = Fn.linear(xt, torch.from_numpy(np.asarray(w1, np.float64)))
    u = Fn.linear(xt, torch.from_numpy(np.asarray(w3, np.float64)))
    return Fn.linear(Fn.silu(g) * u, torch.from_numpy(np.asarray(w2, np.float64))).numpy()


# ----------------------------------------------------------------------- capacity

def test_capacity_named_workloads_closed_form():
    # ceil(1.25*4096*2/16) = ceil(640)   = 640
    # ceil(1.5 *8192*2/8)  = ceil(3072)  = 3072
    # ceil(1.2*16384*2/64) = ceil(614.4) = 615  (a floor would give 614; dropping k, 308)
    assert orc.capacity(4096, 2, 16, 1.25) == 640
    assert orc.capacity(8192, 2, 8, 1.5) == 3072
    assert orc.capacity(16384, 2, 64, 1.2) == 615
    assert orc.capacity(64, 2, 100, None) is None
    assert orc.capacity(64, 2, 8, 0.0) is None
    for c in configs.NAMED:
        C = orc.capacity(c.T, c.k, c.N, c.capacity_factor)
        if c.capacity_factor is None:
            assert C is None
        else:
            assert C >= c.T * c.k / c.N


def test_capacity_page_worked_example():
    g = _kv(GOLDEN / "page_capacity_example.txt")
    batch, seq = int(g["batch"][0]), int(g["seq_len"][0])
    tokens, experts = int(g["num_tokens"][0]), int(g["num_experts"][0])
    assert batch * seq == tokens
    assert tokens // experts == int(g["average_per_expert"][0])
    cf = float(g["capacity_factor"][0])
    assert orc.capacity_page_example_variant(tokens, experts, cf) == int(g["capacity"][0])


# -------------------------------------------------------------------------- top-k

def _brute_force_topk_set(l, k):
    """The unique k-subset S with l_i > l_j, or l_i == l_j and i < j, for every
    i in S and j outside S -- found by enumerating all k-subsets."""
    N = len(l)
    winners = []
    for S in itertools.combinations(range(N), k):
        rest = [j for j in range(N) if j not in S]
        if all(l[i] > l[j] or (l[i] == l[j] and i < j) for i in S for j in rest):
            winners.append(set(S))
    assert len(winners) == 1
    return winners[0]


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(1234)
    for trial in range(2500):
        N = int(rng.integers(1, 9))
        k = int(rng.integers(1, N + 1))
        if trial % 2:
            l = rng.choice([-1.0, -0.5, 0.0, 0.5, 1.0], size=N)   # many exact ties
        else:
            l = rng.standard_normal(N)
        idx = orc.topk_select(l[None, :], k)[0]
        assert set(idx.tolist()) == _brute_force_topk_set(l.tolist(), k)
        for a, b in zip(idx[:-1], idx[1:]):            # slot order: logit desc, id asc
            assert l[a] > l[b] or (l[a] == l[b] and a < b)


def test_topk_all_equal_logits_take_lowest_ids():
    idx = orc.topk_select(np.zeros((3, 7)), 3)
    assert (idx == np.array([0, 1, 2])).all()


# ------------------------------------------------------------------- gate weights

def test_gate_weights_sum_to_one_and_equal_renormalised_probs():
    rng = np.random.default_rng(7)
    l = 3.0 * rng.standard_normal((500, 16))
    for k in (1, 2, 4, 16):
        idx = orc.topk_select(l, k)
        w = orc.gate_weights(l, idx)
        assert np.abs(w.sum(axis=1) - 1.0).max() < 1e-14
        assert (np.diff(w, axis=1) <= 0).all()
        # library softmax over the selected logits
        sel = np.take_along_axis(l, idx, axis=1)
        assert np.abs(w - scipy.special.softmax(sel, axis=1)).max() < 1e-14
        # softmax over all experts, top-k on the probabilities, renormalise
        p = scipy.special.softmax(l, axis=1)
        psel = np.take_along_axis(p, idx, axis=1)
        assert np.abs(w - psel / psel.sum(axis=1, keepdims=True)).max() < 1e-14


def test_full_softmax_matches_library():
    rng = np.random.default_rng(8)
    l = 5.0 * rng.standard_normal((100, 64))
    assert np.abs(orc.full_softmax(l) - scipy.special.softmax(l, axis=1)).max() < 1e-15


def test_router_logits_match_torch():
    rng = np.random.default_rng(9)
    x, wr, b = rng.standard_normal((40, 96)), rng.standard_normal((96, 12)), rng.standard_normal(12)
    ref = (torch.from_numpy(x) @ torch.from_numpy(wr) + torch.from_numpy(b)).numpy()
    assert np.abs(orc.router_logits(x, wr, b) - ref).max() < 1e-12
    assert np.abs(orc.router_logits(x, wr) - (ref - b)).max() < 1e-12


# ------------------------------------------------------------------------ aux loss

@pytest.mark.parametrize("N,k", [(8, 2), (16, 2), (64, 2), (100, 2), (8, 8), (5, 1)])
def test_aux_is_one_for_a_zero_router(N, k):
    # Every P_e = 1/N exactly, so aux = N * sum_e f_e / N = sum_e f_e = 1 for any f.
    x = np.random.default_rng(0).standard_normal((33, 24))
    r = orc.route(x, np.zeros((24, N)), None, k, None)
    assert abs(r["aux_loss"] - 1.0) < 1e-14


@pytest.mark.parametrize("N,k,cycles", [(8, 2, 3), (16, 2, 2), (6, 3, 4)])
def test_aux_is_one_for_cyclic_uniform_routing(N, k, cycles):
    # H = N, W_r = I and x_t = roll(v, t): over whole cycles every expert is chosen
    # T*k/N times and the mean probability of every expert is 1/N.
    v = np.linspace(-1.0, 2.0, N) ** 3
    x = np.stack([np.roll(v, t) for t in range(N * cycles)])
    r = orc.route(x, np.eye(N), None, k, None)
    assert (r["expert_counts"] == N * cycles * k // N).all()
    assert abs(r["aux_loss"] - 1.0) < 1e-13


@pytest.mark.parametrize("N,k,B", [(8, 2, 3.0), (64, 2, 2.0), (10, 4, 0.7)])
def test_aux_one_hot_expert_closed_form(N, k, B):
    # W_r = 0 and bias (B,0,...,0): every token picks experts 0..k-1 (ties go to the
    # lower ids), f_e = 1/k for e < k, P_0 = e^B/(e^B+N-1), P_e = 1/(e^B+N-1), so
    # aux = (N/k) * (e^B + k - 1) / (e^B + N - 1).
    bias = np.zeros(N)
    bias[0] = B
    x = np.random.default_rng(1).standard_normal((50, 16))
    r = orc.route(x, np.zeros((16, N)), bias, k, None)
    assert (r["topk_idx"] == np.arange(k)).all()
    expect = (N / k) * (math.exp(B) + k - 1) / (math.exp(B) + N - 1)
    assert abs(r["aux_loss"] - expect) < 1e-13


def test_aux_uses_counts_before_capacity():
    cfg = configs.TINY_F32
    inp = inputs.make_inputs(cfg, with_experts=False)
    free = orc.route(inp.x, inp.w_router, None, 2, None)
    tight = orc.route(inp.x, inp.w_router, None, 2, 0.05)
    assert tight["drop_mask"].sum() > 0
    assert tight["aux_loss"] == free["aux_loss"]


# ----------------------------------------------------------------------- capacity

@pytest.mark.parametrize("cf", [0.05, 0.5, 1.0, 1.25, 2.0, None])
def test_capacity_invariants(cf):
    rng = np.random.default_rng(11)
    T, H, N, k = 300, 32, 8, 2
    x = rng.standard_normal((T, H))
    wr = 0.3 * rng.standard_normal((H, N))
    bias = np.linspace(0.0, 1.5, N)                     # skewed: some experts overflow
    r = orc.route(x, wr, bias, k, cf)
    C, idx, drop = r["capacity"], r["topk_idx"], r["drop_mask"]
    counts, kept = r["expert_counts"], r["kept_counts"]
    if cf is None:
        assert C is None and drop.sum() == 0 and (kept == counts).all()
        return
    assert (kept == np.minimum(counts, C)).all()
    assert drop.sum() == np.maximum(counts - C, 0).sum()
    for e in range(N):
        # tokens routed to e, in token order; the first C of them are the kept ones
        tok = [t for t in range(T) for s in range(k) if idx[t, s] == e]
        kept_tok = [t for t in range(T) for s in range(k) if idx[t, s] == e and not drop[t, s]]
        assert kept_tok == tok[:C]


# ----------------------------------------------------------------------- expert FFN

def test_silu_against_library_sigmoid():
    z = np.linspace(-30.0, 30.0, 601)
    assert np.abs(orc.silu(z) - z * scipy.special.expit(z)).max() < 1e-14
    assert orc.silu(np.array([0.0]))[0] == 0.0


def test_swiglu_orientation_with_one_hot_weights():
    # W1[a,b] = 1, W3[a,c] = 1, W2[d,a] = 1 and nothing else: the only non-zero output
    # is y[d] = silu(x[b]) * x[c]. A transposed weight, swapped W1/W3 or a missing
    # factor gives a different position or value.
    H, F = 7, 5
    a, b, c, d = 3, 1, 6, 2
    w1 = np.zeros((F, H)); w1[a, b] = 1.0
    w3 = np.zeros((F, H)); w3[a, c] = 1.0
    w2 = np.zeros((H, F)); w2[d, a] = 1.0
    x = np.random.default_rng(3).standard_normal((4, H))
    y = orc.swiglu_expert(x, w1, w3, w2)
    expect = np.zeros((4, H))
    expect[:, d] = x[:, b] * scipy.special.expit(x[:, b]) * x[:, c]
    assert np.abs(y - expect).max() < 1e-15


def test_swiglu_matches_torch_float64():
    rng = np.random.default_rng(4)
    H, F = 96, 160
    x = rng.standard_normal((20, H))
    w1, w3 = rng.standard_normal((F, H)) / 10, rng.standard_normal((F, H)) / 10
    w2 = rng.standard_normal((H, F)) / 12
    ref = _torch_swiglu(x, w1, w3, w2)
    assert np.abs(orc.swiglu_expert(x, w1, w3, w2) - ref).max() < 1e-12 * np.abs(ref).max()


# ----------------------------------------------------------------------- the layer

def test_k_equals_n_without_capacity_is_the_dense_softmax_mixture():
    cfg = configs.TINY_F32.with_(k=8)
    inp = inputs.make_inputs(cfg)
    x, wr = inp.x.astype(np.float64), inp.w_router.astype(np.float64)
    res = orc.moe_forward(x, wr, None, inp.w1, inp.w3, inp.w2, cfg.k, None)
    p = scipy.special.softmax(x @ wr, axis=1)
    dense = sum(p[:, e:e + 1] * _torch_swiglu(x, inp.w1[e], inp.w3[e], inp.w2[e])
                for e in range(cfg.N))
    assert np.abs(res.out - dense).max() < 1e-12 * np.abs(dense).max()


def test_single_expert_is_a_dense_swiglu_ffn():
    cfg = configs.TINY_F32.with_(N=1, k=1)
    inp = inputs.make_inputs(cfg)
    res = orc.moe_forward(inp.x, inp.w_router, None, inp.w1, inp.w3, inp.w2, 1, None)
    ref = _torch_swiglu(inp.x, inp.w1[0], inp.w3[0], inp.w2[0])
    assert (res.topk_w == 1.0).all()
    assert np.abs(res.out - ref).max() < 1e-12 * np.abs(ref).max()


def test_dropped_slots_give_zero_and_kept_weights_are_not_renormalised():
    # H = N = 4, W_r = I: token 0 -> experts {0,1}, token 1 -> {1,2}, token 2 -> {0,1}.
    # C = ceil(0.5*3*2/4) = 1: expert 1 keeps token 0 only, expert 0 keeps token 0.
    N = 4
    x = np.array([[3.0, 2.0, 0.0, -1.0],
                  [0.0, 3.0, 2.0, -1.0],
                  [3.0, 2.0, 0.0, -1.0]])
    rng = np.random.default_rng(5)
    F = 6
    w1, w3 = rng.standard_normal((N, F, N)), rng.standard_normal((N, F, N))
    w2 = rng.standard_normal((N, N, F))
    res = orc.moe_forward(x, np.eye(N), None, w1, w3, w2, 2, 0.5)
    assert res.capacity == 1
    assert res.topk_idx.tolist() == [[0, 1], [1, 2], [0, 1]]
    assert res.drop_mask.tolist() == [[0, 0], [1, 0], [1, 1]]
    assert (res.out[2] == 0.0).all()                     # every slot dropped -> 0
    w_kept = math.exp(-1.0) / (1.0 + math.exp(-1.0))     # softmax of logits (3, 2), slot 1
    assert abs(res.topk_w[1, 1] - w_kept) < 1e-15
    y_e2 = _torch_swiglu(x[1:2], w1[2], w3[2], w2[2])[0]
    assert np.abs(res.out[1] - w_kept * y_e2).max() < 1e-12 * np.abs(y_e2).max()


def test_token_sample_rows_equal_full_rows():
    cfg = configs.TINY_F32.with_(capacity_factor=0.9)
    inp = inputs.make_inputs(cfg)
    full = orc.moe_forward(inp.x, inp.w_router, None, inp.w1, inp.w3, inp.w2, 2, 0.9)
    sample = np.array([0, 5, 17, 63])
    part = orc.moe_forward(inp.x, inp.w_router, None, inp.w1, inp.w3, inp.w2, 2, 0.9,
                           token_sample=sample)
    # same arithmetic; only the BLAS blocking over a different row count may differ
    assert np.abs(part.out - full.out[sample]).max() < 1e-13 * np.abs(full.out).max()


def test_empty_batch():
    res = orc.moe_forward(np.zeros((0, 8)), np.zeros((8, 4)), None, np.zeros((4, 6, 8)),
                          np.zeros((4, 6, 8)), np.zeros((4, 8, 6)), 2, 1.25)
    assert res.out.shape == (0, 8) and res.aux_loss == 0.0
    assert res.expert_counts.sum() == 0 and res.capacity == 0


def test_active_fraction_page_values():
    g = _kv(GOLDEN / "page_active_fractions.txt")
    rng = np.random.default_rng(6)
    for k, E, frac in zip(g["k"], g["experts"], g["fraction"]):
        k, E, frac = int(k), int(E), float(frac)
        assert k / E == frac
        l = rng.standard_normal((200, E))
        assert orc.active_fraction(orc.topk_select(l, k), E) == frac


def test_near_tie_detection():
    l = np.array([[1.0, 0.99995, 0.2],       # 2nd/3rd fine, 1st/2nd order tie
                  [1.0, 0.5, 0.49995],       # set tie at k = 2
                  [1.0, 0.5, 0.4998]])       # no tie
    set_ties, order_ties = orc.near_tie_tokens(l, 2)
    assert set_ties.tolist() == [1]
    assert order_ties.tolist() == [0]


# ------------------------------------------------------------------ input recipe

def test_bf16_rounding_is_round_to_nearest_even():
    one = np.float32(1.0)
    half_ulp = np.float32(2.0 ** -8)
    vals = np.array([one, one + half_ulp, one + 3 * half_ulp, -one - half_ulp], np.float32)
    bits = inputs.f32_to_bf16_bits(vals)
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xBF80]
    r = np.random.default_rng(2).standard_normal(10000).astype(np.float32)
    ref = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (inputs.f32_to_bf16_bits(r) == ref).all()
    assert (inputs.bf16_bits_to_f32(ref) == torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy()).all()


def test_zipf_bias_profile():
    inp = inputs.make_inputs(configs.FINEGRAINED_T16384.with_(T=8, H=64, F=128),
                             with_experts=False)
    b = np.sort(inp.router_bias)[::-1]
    assert b[0] == np.float32(2.0)
    assert np.allclose(b, 2.0 * np.arange(1, 65, dtype=np.float64) ** -1.1, rtol=1e-6)
