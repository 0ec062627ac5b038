"""The seeded input recipe that feeds both the CUDA path and the oracle: reproducible
per seed, the stated distributions, shared experts that extend the routed ones, per-rank
batches over shared weights, padded-sequence masks, and the exact-logit inputs that the
exact rerouting comparisons rely on. CPU only."""
import numpy as np
import pytest

from mixture_experts_layer_102_b300 import configs, inputs

SMALL_BF16 = configs.MoEConfig("inputs_bf16", 512, 256, 8, 2, 384, 1.25, "bf16", seed=5)


def _arrays(inp):
    return [inp.x, inp.w_router, inp.w1, inp.w3, inp.w2]


def test_same_seed_same_inputs_other_seed_other_inputs():
    a = inputs.make_inputs(SMALL_BF16)
    b = inputs.make_inputs(SMALL_BF16)
    for u, v in zip(_arrays(a), _arrays(b)):
        assert u.dtype == np.uint16 and (u == v).all()
    c = inputs.make_inputs(SMALL_BF16.with_(seed=6))
    for u, v in zip(_arrays(a), _arrays(c)):
        assert (u != v).any()


def test_shapes_and_storage_types():
    inp = inputs.make_inputs(SMALL_BF16)
    T, H, N, F = SMALL_BF16.T, SMALL_BF16.H, SMALL_BF16.N, SMALL_BF16.F
    assert inp.x.shape == (T, H) and inp.w_router.shape == (H, N)
    assert inp.w1.shape == (N, F, H) and inp.w3.shape == (N, F, H) and inp.w2.shape == (N, H, F)
    assert inp.router_bias is None
    f32 = inputs.make_inputs(configs.TINY_F32)
    assert f32.x.dtype == np.float32 and f32.w1.dtype == np.float32


@pytest.mark.parametrize("name,std", [("x", 1.0), ("w_router", 0.02), ("w1", 256 ** -0.5),
                                      ("w3", 256 ** -0.5), ("w2", 384 ** -0.5)])
def test_draws_have_the_stated_spread(name, std):
    v = inputs.make_inputs(SMALL_BF16).values(name).astype(np.float64)
    # within five standard errors: std/std_target has s.e. 1/sqrt(2n), the mean std/sqrt(n)
    n = v.size
    assert abs(v.std() / std - 1.0) < 5.0 / np.sqrt(2 * n), (name, v.std(), std)
    assert abs(v.mean()) < 5.0 * std / np.sqrt(n)


def test_bf16_storage_holds_the_rounded_draws():
    # widening the stored bits and rounding again changes nothing
    inp = inputs.make_inputs(SMALL_BF16)
    v = inp.values("w1")
    assert (inputs.f32_to_bf16_bits(v) == inp.w1).all()


def test_shared_experts_extend_the_routed_experts():
    base = inputs.make_inputs(SMALL_BF16)
    sh = inputs.make_inputs(SMALL_BF16, n_shared=2)
    N = SMALL_BF16.N
    for name in ("w1", "w3", "w2"):
        a, b = getattr(base, name), getattr(sh, name)
        assert b.shape[0] == N + 2 and (b[:N] == a).all()
    assert (sh.x == base.x).all() and (sh.w_router == base.w_router).all()


def test_ranks_draw_their_own_batch_over_the_same_weights():
    r0 = inputs.make_inputs(SMALL_BF16, rank=0)
    r1 = inputs.make_inputs(SMALL_BF16, rank=1)
    r2 = inputs.make_inputs(SMALL_BF16, rank=2)
    assert (r0.x != r1.x).any() and (r1.x != r2.x).any()
    for name in ("w_router", "w1", "w3", "w2"):
        assert (getattr(r0, name) == getattr(r1, name)).all()
    assert (inputs.make_x(SMALL_BF16, rank=1) == r1.x).all()


@pytest.mark.parametrize("T,seq_len", [(1000, 50), (37, 8), (64, 64), (5, 100)])
def test_valid_mask_is_a_prefix_of_each_sequence(T, seq_len):
    m = inputs.make_valid_mask(T, seq_len, seed=11)
    assert m.shape == (T,) and m.dtype == np.uint8 and set(np.unique(m)) <= {0, 1}
    for s0 in range(0, T, seq_len):
        seq = m[s0:s0 + seq_len]
        L = int(seq.sum())
        assert (seq[:L] == 1).all() and (seq[L:] == 0).all()  # real tokens first
    assert (inputs.make_valid_mask(T, seq_len, seed=11) == m).all()
    assert inputs.make_valid_mask(0, seq_len, seed=11).shape == (0,)


def test_valid_mask_lengths_cover_the_whole_range():
    m = inputs.make_valid_mask(200 * 16, 16, seed=3)
    lengths = m.reshape(200, 16).sum(axis=1)
    assert lengths.min() == 0 and lengths.max() == 16  # empty and full sequences occur


@pytest.mark.parametrize("zipf", [False, True])
def test_separated_inputs_give_logits_on_a_1_128_grid(zipf):
    cfg = configs.MoEConfig("sep", 300, 128, 24, 2, 128, 1.0, "bf16", seed=9, zipf_bias=zipf)
    inp = inputs.make_separated_inputs(cfg)
    x = inp.values("x").astype(np.float64)
    wr = inp.values("w_router").astype(np.float64)
    logits = x @ wr
    if zipf:
        logits = logits + inp.router_bias.astype(np.float64)
    scaled = logits * 128.0
    assert (scaled == np.round(scaled)).all()
    # each token's routed part is a permutation of 0, 1/64, ..., (N-1)/64: no equal pair
    routed = np.sort(x[:, :cfg.N], axis=1)
    assert (routed == np.arange(cfg.N) / 64.0).all()
    # the experts' weights are the ordinary draws
    assert (inp.w1 == inputs.make_inputs(cfg).w1).all()


def test_separated_inputs_refuse_too_many_experts():
    with pytest.raises(ValueError):
        inputs.make_separated_inputs(configs.MoEConfig("sep", 8, 64, 65, 2, 64, 1.0, "bf16"))
