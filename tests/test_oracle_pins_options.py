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
