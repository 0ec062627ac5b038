"""Parity of the layer options (shared experts, the GELU expert, a valid-token mask,
the KL and variance balance losses) through moe_forward_ex / moe_route_ex with the
fp64 oracle on the same seeded inputs.

Criteria: those of the base parity tests, taken over the valid tokens, plus
* padding tokens: topk_idx -1, topk_w 0, every slot dropped, output exactly 0;
* with shared experts a token whose routed slots were all dropped still gets the
  shared experts' output, so the exact-zero check of such rows applies only
  without them;
* aux_kl within 1e-6 relative of the oracle's value: both sides take the logarithms
  of the same integer counts in double (when a near tie moved a slot, the reference
  is the oracle's KL of the GPU's own counts);
* aux_std2 within 2e-4 relative (plus 1e-12 absolute) of the oracle's value: the GPU
  sums (P - 1/N)^2 of fp32 probabilities, in fp32 inside a block and in double
  across blocks, and its probabilities differ from the fp64 ones by the router's
  accumulation rounding (about 1e-6 relative).
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
import parity_report
from mixture_experts_layer_102_b300 import configs, inputs, moe
from mixture_experts_layer_102_b300.configs import MoEConfig

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}
TOL_AUX = 1e-5
TOL_W = 1e-5
TOL_KL = 1e-6
TOL_STD2 = 2e-4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_102_b300 import build
    build.build(quiet=True)


def _rel_err(y, r):
    if r.size == 0:
        return 0.0
    rms = np.sqrt(np.mean(r * r))
    return float(np.max(np.abs(y - r) / (np.abs(r) + rms + 1e-30)))


def _max_ratio(y, r):
    """max |y - r| / max |r|, reported beside the gated metric."""
    if r.size == 0 or not np.abs(r).max() > 0:
        return 0.0
    return float(np.abs(y - r).max() / np.abs(r).max())


def run_opts(cfg, inp, n_shared=0, activation="swiglu", mask=None, reroute=False,
             losses=True):
    c = moe.cfg_from(cfg)
    dev = moe.to_device(inp)
    vm = None if mask is None else torch.from_numpy(mask).cuda()
    kl = torch.full((1,), -7.0, device="cuda") if losses else None
    s2 = torch.full((1,), -7.0, device="cuda") if losses else None
    opts = moe.Options(n_shared, activation, vm, kl, s2, reroute)
    ws = moe.make_workspace(c, options=opts)
    routing = moe.new_routing(c)
    w3 = None if activation == "gelu" else dev.w3
    out = moe.forward(c, dev.x, dev.w_router, dev.router_bias, dev.w1, w3, dev.w2,
                      workspace=ws, routing=routing, options=opts)
    assert moe.get_status(ws) == 0
    g = {k: getattr(routing, k).cpu().numpy() for k in
         ("topk_idx", "topk_w", "aux_loss", "drop_mask", "expert_counts", "kept_counts")}
    g["out"] = out.float().cpu().numpy()
    g["aux_kl"] = float(kl.item()) if losses else None
    g["aux_std2"] = float(s2.item()) if losses else None
    return g, (c, dev, ws, opts)


def oracle_opts(cfg, inp, n_shared=0, activation="swiglu", mask=None, token_sample=None,
                reroute=False):
    x, wr = inp.values("x"), inp.values("w_router")
    return orc.moe_forward(x, wr, inp.router_bias, inp.values("w1"),
                           None if activation == "gelu" else inp.values("w3"),
                           inp.values("w2"), cfg.k, cfg.capacity_factor,
                           token_sample=token_sample, n_shared=n_shared,
                           activation=activation, valid_mask=mask, reroute=reroute)


def compare_opts(cfg, g, ref, mask, n_shared):
    T, k, N = cfg.T, cfg.k, cfg.N
    valid = np.ones(T, bool) if mask is None else mask.astype(bool)
    pad = ~valid
    assert (g["topk_idx"][pad] == -1).all() and (g["topk_w"][pad] == 0).all()
    assert (g["drop_mask"][pad] == 1).all()
    v = np.nonzero(valid)[0]
    idx_g = g["topk_idx"].astype(np.int64)
    idx_r = ref.topk_idx
    set_ties = set(ref.near_tie_set.tolist())
    order_ties = set(ref.near_tie_order.tolist())
    same_set = (np.sort(idx_g, axis=1) == np.sort(idx_r, axis=1)).all(axis=1)
    flipped = np.nonzero(~same_set)[0]
    assert set(flipped.tolist()) <= set_ties, f"tokens routed differently: {flipped[:10]}"
    reordered = np.nonzero(same_set & (idx_g != idx_r).any(axis=1))[0]
    assert set(reordered.tolist()) <= order_ties, f"slot order differs: {reordered[:10]}"
    for t in flipped:
        kth = np.sort(ref.logits[t])[::-1][k - 1]
        assert (ref.logits[t, idx_g[t]] >= kth - orc.NEAR_TIE_MARGIN).all()

    exact = (idx_g == idx_r).all(axis=1) & valid
    assert np.abs(g["topk_w"][exact] - ref.topk_w[exact]).max(initial=0.0) <= TOL_W
    assert abs(float(g["aux_loss"][0]) - ref.aux_loss) <= TOL_AUX, (g["aux_loss"], ref.aux_loss)

    C = ref.capacity
    counts_g = np.bincount(idx_g[v].ravel(), minlength=N)
    assert (g["expert_counts"] == counts_g).all()
    if len(flipped) == 0:
        assert (g["expert_counts"] == ref.expert_counts).all()
        assert (g["drop_mask"] == ref.drop_mask).all()
        assert (g["kept_counts"] == ref.kept_counts).all()
        kl_ref = ref.aux_kl
    else:
        # the GPU's capacity decisions must be the valid ones for its own routing:
        # each expert keeps its first C slots in token order
        sel_g, drop_g = idx_g[v], g["drop_mask"][v]
        for e in range(N):
            kept = drop_g[sel_g == e] == 0
            want = np.arange(kept.size) < (C if C is not None else kept.size)
            assert (kept == want).all()
        kl_ref = orc.aux_kl_uniform(idx_g[v], N, k)
    if C is not None:
        assert (g["kept_counts"] == np.minimum(counts_g, C)).all()
    else:
        assert g["drop_mask"][v].sum() == 0

    if g["aux_kl"] is None:  # the optional losses were not asked for
        pass
    elif math.isinf(kl_ref):
        assert g["aux_kl"] == math.inf
    else:
        assert abs(g["aux_kl"] - kl_ref) <= TOL_KL * max(1.0, abs(kl_ref)), (g["aux_kl"], kl_ref)
    if g["aux_std2"] is None:
        pass
    elif math.isnan(ref.aux_std2):
        assert math.isnan(g["aux_std2"])
    else:
        assert abs(g["aux_std2"] - ref.aux_std2) <= TOL_STD2 * abs(ref.aux_std2) + 1e-12, \
            (g["aux_std2"], ref.aux_std2)

    rows = ref.tokens
    keep = np.ones(len(rows), dtype=bool)
    if len(flipped):
        touched = set()
        for t in flipped:
            touched |= set(idx_g[t].tolist()) ^ set(idx_r[t].tolist())
        keep = np.array([not (set(idx_r[t].tolist()) & touched) for t in rows])
    assert (g["out"][rows[~valid[rows]]] == 0).all()
    dropped_all = ref.drop_mask[rows].all(axis=1) & valid[rows]
    live = keep & valid[rows] & (~dropped_all if n_shared == 0 else True)
    err = _rel_err(g["out"][rows[live]], ref.out[live])
    info = dict(err=err, max_ratio=_max_ratio(g["out"][rows[live]], ref.out[live]),
                near_tie_set=len(set_ties), near_tie_order=len(order_ties),
                flipped=len(flipped), reordered=len(reordered), valid=int(valid.sum()))
    parity_report.record(f"{cfg.name} (S={n_shared})", **info)
    assert err <= TOL[cfg.dtype], f"output relative error {err:.3e} > {TOL[cfg.dtype]}"
    if n_shared == 0:
        assert (g["out"][rows[dropped_all & keep]] == 0).all()
    return info


def check_opts(cfg, n_shared=0, activation="swiglu", seq_len=None, token_sample=None,
               losses=True):
    inp = inputs.make_inputs(cfg, n_shared=n_shared)
    mask = None if seq_len is None else inputs.make_valid_mask(cfg.T, seq_len, cfg.seed)
    g, _ = run_opts(cfg, inp, n_shared, activation, mask, losses=losses)
    ref = oracle_opts(cfg, inp, n_shared, activation, mask, token_sample)
    return compare_opts(cfg, g, ref, mask, n_shared)


# (workload, shared experts, activation, sequence length of the padding mask or None)
# bf16 layers of 32 or more tiles of 128 tokens run the fused router + routing kernel
CASES = [
    (MoEConfig("bf16_fused_n256_k8_t4000", 4000, 128, 256, 8, 64, 1.5, "bf16", seed=38), 0,
     "swiglu", None),
    (MoEConfig("bf16_fused_n16_t6000", 6000, 128, 16, 2, 64, 1.25, "bf16", seed=49), 0,
     "swiglu", None),
    (MoEConfig("bf16_fused_n48_k3_t7001_masked_shared", 7001, 64, 48, 3, 64, 1.0, "bf16",
               seed=50, zipf_bias=True), 1, "swiglu", 500),
    (MoEConfig("bf16_fused_n1_k1_t4096", 4096, 128, 1, 1, 64, None, "bf16", seed=39), 0,
     "swiglu", None),
    # few experts over 40 blocks with shared experts and capacity drops (the optional
    # losses asked for here keep the block finish; see the one-warp test below)
    (MoEConfig("bf16_fused_n5_t5000", 5000, 128, 5, 2, 64, 1.1, "bf16", seed=52,
               zipf_bias=True), 2, "swiglu", None),
    (MoEConfig("bf16_fused_k32_n64_masked_shared", 4100, 64, 64, 32, 64, 0.9, "bf16", seed=40,
               zipf_bias=True), 2, "gelu", 300),
    (configs.TINY_F32.with_(name="f32_shared2_tight", capacity_factor=0.6), 2, "swiglu", None),
    (configs.TINY_F32.with_(name="f32_gelu"), 0, "gelu", None),
    (configs.TINY_F32.with_(name="f32_masked", capacity_factor=1.0), 0, "swiglu", 16),
    (MoEConfig("f32_masked_shared_gelu", 300, 192, 5, 2, 320, 0.9, "f32", seed=31), 1, "gelu", 50),
    (MoEConfig("bf16_shared1_ragged", 1000, 256, 8, 2, 384, 1.25, "bf16", seed=21), 1, "swiglu",
     None),
    (MoEConfig("bf16_gelu_ragged", 1000, 256, 8, 2, 384, 1.25, "bf16", seed=22), 0, "gelu", None),
    (MoEConfig("bf16_gelu_edge_h320_f192", 777, 320, 6, 2, 192, 1.1, "bf16", seed=23), 0, "gelu",
     None),
    (MoEConfig("bf16_masked_ragged", 1000, 256, 8, 2, 384, 1.0, "bf16", seed=24), 0, "swiglu",
     128),
    (MoEConfig("bf16_masked_shared2_gelu", 1500, 256, 16, 2, 256, 1.25, "bf16", seed=25), 2,
     "gelu", 200),
    # 256-row tiles on CTA pairs
    (MoEConfig("bf16_pair_shared1", 3000, 256, 4, 2, 384, 1.25, "bf16", seed=26), 1, "swiglu",
     None),
    (MoEConfig("bf16_pair_gelu_masked", 4096, 128, 4, 2, 128, 1.02, "bf16", seed=27,
               zipf_bias=True), 0, "gelu", 512),
    # GEMM1 (GELU) on CTA pairs, GEMM2 on single CTAs
    (MoEConfig("bf16_mixed_tiles_gelu", 2048, 256, 8, 2, 384, 1.25, "bf16", seed=37), 0, "gelu",
     None),
    (MoEConfig("bf16_zipf_masked_shared8", 2048, 128, 64, 2, 128, 1.2, "bf16", seed=28,
               zipf_bias=True), 8, "swiglu", 100),
    # k + n_shared = 40 slots per token
    (MoEConfig("bf16_k32_shared8", 96, 64, 64, 32, 64, None, "bf16", seed=29), 8, "swiglu", 16),
    # five tokens per warp in the routing decisions (ranks kept in memory past four)
    (MoEConfig("bf16_t100000_masked_shared1", 100000, 64, 8, 2, 64, 1.25, "bf16", seed=30), 1,
     "swiglu", 300),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_options_elementwise(case):
    cfg, n_shared, act, seq_len = case
    check_opts(cfg, n_shared, act, seq_len)


# Shared experts without a mask or the optional losses: the routing kernel finishes in
# one warp, on the fused path (4 lanes per expert over ragged ranges of 40 blocks) and
# on the two-launch path (22 blocks of 32 tokens).
WARP_FINISH_SHARED = [
    (MoEConfig("bf16_fused_n5_t5000_s2_warp_finish", 5000, 128, 5, 2, 64, 1.1, "bf16",
               seed=53, zipf_bias=True), 2),
    (MoEConfig("bf16_select_n6_t700_s1_warp_finish", 700, 128, 6, 2, 128, 1.1, "bf16",
               seed=54), 1),
]


@pytest.mark.parametrize("case", WARP_FINISH_SHARED, ids=lambda c: c[0].name)
def test_shared_experts_with_the_one_warp_finish(case):
    cfg, n_shared = case
    plan = moe.describe(moe.cfg_from(cfg), moe.Options(n_shared=n_shared),
                        has_bias=cfg.zipf_bias)
    assert plan["routing_warp_finish"] == 1
    check_opts(cfg, n_shared, "swiglu", None, losses=False)


def test_bench_shape_with_every_option_sampled():
    cfg = configs.BF16_T4096
    inp = inputs.make_inputs(cfg, n_shared=1)
    mask = inputs.make_valid_mask(cfg.T, 1024, cfg.seed)
    g, _ = run_opts(cfg, inp, 1, "gelu", mask)
    sample = np.random.default_rng(5).choice(cfg.T, size=192, replace=False)
    ref = oracle_opts(cfg, inp, 1, "gelu", mask, np.sort(sample))
    compare_opts(cfg, g, ref, mask, 1)


@pytest.mark.parametrize("c", [configs.BF16_T4096, configs.FINEGRAINED_T16384],
                         ids=lambda c: c.name)
def test_losses_on_named_workloads(c):
    inp = inputs.make_inputs(c, with_experts=False)
    dev_x = moe.to_torch(inp.x, c.dtype).cuda()
    dev_wr = moe.router_weight_to_device(inp.w_router, c.dtype)
    bias = None if inp.router_bias is None else torch.from_numpy(inp.router_bias).cuda()
    cc = moe.cfg_from(c)
    kl = torch.zeros(1, device="cuda")
    s2 = torch.zeros(1, device="cuda")
    opts = moe.Options(aux_kl=kl, aux_std2=s2)
    ws = moe.make_workspace(cc, options=opts)
    r = moe.route(cc, dev_x, dev_wr, bias, workspace=ws, options=opts)
    assert moe.get_status(ws) == 0
    ref = orc.route(inp.values("x"), inp.values("w_router"), inp.router_bias, c.k,
                    c.capacity_factor)
    idx_g = r.topk_idx.cpu().numpy().astype(np.int64)
    kl_ref = orc.aux_kl_uniform(idx_g, c.N, c.k)   # of the GPU's own counts
    assert abs(kl.item() - kl_ref) <= TOL_KL * max(1.0, abs(kl_ref))
    assert abs(s2.item() - ref["aux_std2"]) <= TOL_STD2 * abs(ref["aux_std2"]) + 1e-12
    assert abs(r.aux_loss.item() - ref["aux_loss"]) <= TOL_AUX


def test_all_padding_gives_zeros():
    cfg = MoEConfig("bf16_all_padding", 500, 128, 8, 2, 128, 1.25, "bf16", seed=32)
    inp = inputs.make_inputs(cfg, n_shared=1)
    mask = np.zeros(cfg.T, np.uint8)
    g, _ = run_opts(cfg, inp, 1, "swiglu", mask)
    assert (g["out"] == 0).all() and (g["topk_idx"] == -1).all() and (g["drop_mask"] == 1).all()
    assert float(g["aux_loss"][0]) == 0.0 and g["aux_kl"] == 0.0 and g["aux_std2"] == 0.0
    assert g["expert_counts"].sum() == 0 and g["kept_counts"].sum() == 0


def test_single_valid_token_single_expert_variance_is_nan():
    # T_valid * N = 1: the unbiased variance of one probability is undefined
    cfg = MoEConfig("f32_one_valid", 4, 64, 1, 1, 64, None, "f32", seed=33)
    inp = inputs.make_inputs(cfg)
    mask = np.array([0, 0, 1, 0], np.uint8)
    g, _ = run_opts(cfg, inp, 0, "swiglu", mask)
    ref = oracle_opts(cfg, inp, 0, "swiglu", mask)
    assert math.isnan(ref.aux_std2) and math.isnan(g["aux_std2"])
    compare_opts(cfg, g, ref, mask, 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_base_options_are_bit_identical_to_the_base_call(dtype):
    cfg = MoEConfig(f"{dtype}_base_vs_ex", 1200, 128, 8, 2, 192, 1.1, dtype, seed=34)
    inp = inputs.make_inputs(cfg)
    dev = moe.to_device(inp)
    c = moe.cfg_from(cfg)
    base = moe.forward(c, dev.x, dev.w_router, dev.router_bias, dev.w1, dev.w3, dev.w2)
    r_base = moe.new_routing(c)
    moe.forward(c, dev.x, dev.w_router, dev.router_bias, dev.w1, dev.w3, dev.w2, routing=r_base)
    # default options, and an all-valid mask, go through the *_ex path
    for mask in (None, torch.ones(cfg.T, dtype=torch.uint8, device="cuda")):
        r = moe.new_routing(c)
        ex = moe.forward(c, dev.x, dev.w_router, dev.router_bias, dev.w1, dev.w3, dev.w2,
                         routing=r, options=moe.Options(valid_mask=mask))
        assert torch.equal(ex, base)
        for name in ("topk_idx", "topk_w", "aux_loss", "drop_mask", "expert_counts",
                     "kept_counts"):
            assert torch.equal(getattr(r, name), getattr(r_base, name)), name


def test_route_ex_matches_forward_ex():
    cfg = MoEConfig("bf16_route_ex", 1500, 256, 16, 2, 256, 1.0, "bf16", seed=35)
    inp = inputs.make_inputs(cfg, n_shared=2)
    mask = inputs.make_valid_mask(cfg.T, 100, cfg.seed)
    g, (c, dev, ws, opts) = run_opts(cfg, inp, 2, "swiglu", mask)
    kl2 = torch.zeros(1, device="cuda")
    s22 = torch.zeros(1, device="cuda")
    ropts = moe.Options(2, "swiglu", opts.valid_mask, kl2, s22)
    r = moe.route(c, dev.x, dev.w_router, dev.router_bias, workspace=ws, options=ropts)
    assert moe.get_status(ws) == 0
    for name in ("topk_idx", "topk_w", "aux_loss", "drop_mask", "expert_counts", "kept_counts"):
        assert (getattr(r, name).cpu().numpy() == g[name]).all(), name
    assert kl2.item() == g["aux_kl"] and s22.item() == g["aux_std2"]


def test_repeat_calls_with_options_are_bit_identical():
    cfg = MoEConfig("bf16_repeat_opts", 2000, 256, 8, 2, 256, 1.25, "bf16", seed=36)
    inp = inputs.make_inputs(cfg, n_shared=1)
    mask = inputs.make_valid_mask(cfg.T, 256, cfg.seed)
    g1, (c, dev, ws, opts) = run_opts(cfg, inp, 1, "gelu", mask)
    out2 = moe.forward(c, dev.x, dev.w_router, dev.router_bias, dev.w1, None, dev.w2,
                       workspace=ws, options=opts)
    assert moe.get_status(ws) == 0
    assert (out2.float().cpu().numpy() == g1["out"]).all()


def test_bad_options_are_refused():
    cfg = configs.TINY_F32
    inp = inputs.make_inputs(cfg)
    dev = moe.to_device(inp)
    c = moe.cfg_from(cfg)
    with pytest.raises(moe.MoEError):   # the library refuses the option itself
        moe.make_workspace(c, options=moe.Options(n_shared=moe.MOE_MAX_SHARED + 1))
    with pytest.raises(ValueError):
        moe.forward(c, dev.x, dev.w_router, None, dev.w1, dev.w3, dev.w2,
                    options=moe.Options(n_shared=1))   # weights hold only N experts


# ------------------------------------------------------------ overflow rerouting
#
# Inputs with separated router logits (inputs.make_separated_inputs): every logit is
# an exact multiple of 1/128 on both sides, so every routing and rerouting decision
# (including equal logits, broken to the lower id by both) must match exactly.

def compare_reroute(cfg, g, ref, mask, n_shared):
    T = cfg.T
    valid = np.ones(T, bool) if mask is None else mask.astype(bool)
    assert (g["topk_idx"] == ref.topk_idx).all(), "final experts differ"
    assert (g["drop_mask"] == ref.drop_mask).all(), "final drops differ"
    assert (g["expert_counts"] == ref.expert_counts).all()
    assert (g["kept_counts"] == ref.kept_counts).all()
    if ref.capacity is not None:
        assert (g["kept_counts"] <= ref.capacity).all()
    assert np.abs(g["topk_w"] - ref.topk_w).max(initial=0.0) <= TOL_W
    assert abs(float(g["aux_loss"][0]) - ref.aux_loss) <= TOL_AUX
    rows = ref.tokens
    vr = valid[rows]
    dropped_all = ref.drop_mask[rows].all(axis=1) & vr
    live = vr & (~dropped_all if n_shared == 0 else True)
    err = _rel_err(g["out"][rows[live]], ref.out[live])
    info = dict(err=err, max_ratio=_max_ratio(g["out"][rows[live]], ref.out[live]),
                rerouted=int(ref.rerouted.sum()), dropped=int(ref.drop_mask[valid].sum()))
    parity_report.record(f"{cfg.name} (separated logits, rerouting)", **info)
    assert err <= TOL[cfg.dtype], f"output relative error {err:.3e} > {TOL[cfg.dtype]}"
    assert (g["out"][rows[~vr]] == 0).all()
    if n_shared == 0:
        assert (g["out"][rows[dropped_all]] == 0).all()
    return info


def check_reroute(cfg, n_shared=0, activation="swiglu", seq_len=None, token_sample=None):
    inp = inputs.make_separated_inputs(cfg, n_shared=n_shared)
    mask = None if seq_len is None else inputs.make_valid_mask(cfg.T, seq_len, cfg.seed)
    g, _ = run_opts(cfg, inp, n_shared, activation, mask, reroute=True)
    ref = oracle_opts(cfg, inp, n_shared, activation, mask, token_sample, reroute=True)
    info = compare_reroute(cfg, g, ref, mask, n_shared)
    assert info["rerouted"] > 0   # the case exercises rerouting
    return info


REROUTE_CASES = [
    (MoEConfig("bf16_reroute_zipf_n64", 2048, 128, 64, 2, 128, 1.2, "bf16", seed=41,
               zipf_bias=True), 0, "swiglu", None),
    (MoEConfig("bf16_reroute_k4_n32", 1000, 128, 32, 4, 128, 0.8, "bf16", seed=42,
               zipf_bias=True), 0, "swiglu", None),
    (MoEConfig("f32_reroute", 300, 192, 16, 2, 320, 1.0, "f32", seed=43, zipf_bias=True), 0,
     "swiglu", None),
    (MoEConfig("bf16_reroute_uniform", 3000, 128, 16, 2, 128, 1.05, "bf16", seed=46), 0,
     "swiglu", None),
    (MoEConfig("bf16_reroute_k1", 1500, 256, 16, 1, 256, 0.9, "bf16", seed=47, zipf_bias=True),
     0, "swiglu", None),
    # 256-row tiles on CTA pairs
    (MoEConfig("bf16_reroute_pair", 4096, 128, 4, 2, 128, 1.02, "bf16", seed=44,
               zipf_bias=True), 0, "swiglu", None),
    # after the fused routing kernel, with a ragged last tile
    (MoEConfig("bf16_reroute_fused_t5000", 5000, 128, 24, 2, 64, 0.95, "bf16", seed=51,
               zipf_bias=True), 0, "swiglu", None),
    (MoEConfig("bf16_reroute_masked_shared2_gelu", 1500, 256, 16, 2, 256, 1.0, "bf16", seed=48,
               zipf_bias=True), 2, "gelu", 100),
]


@pytest.mark.parametrize("case", REROUTE_CASES, ids=lambda c: c[0].name)
def test_reroute_elementwise(case):
    cfg, n_shared, act, seq_len = case
    check_reroute(cfg, n_shared, act, seq_len)


def test_reroute_many_tokens_per_warp_sampled():
    # 100 000 tokens: five per routing warp; outputs on a seeded sample of rows
    cfg = MoEConfig("bf16_reroute_t100000", 100000, 128, 32, 2, 64, 1.1, "bf16", seed=45,
                    zipf_bias=True)
    sample = np.sort(np.random.default_rng(7).choice(cfg.T, size=3000, replace=False))
    check_reroute(cfg, 1, "swiglu", 500, token_sample=sample)


def test_reroute_without_capacity_changes_nothing():
    cfg = MoEConfig("bf16_reroute_nocap", 700, 128, 8, 2, 128, None, "bf16", seed=49)
    inp = inputs.make_inputs(cfg)
    g0, _ = run_opts(cfg, inp)
    g1, _ = run_opts(cfg, inp, reroute=True)
    for name in ("topk_idx", "topk_w", "drop_mask", "kept_counts", "out"):
        assert (g0[name] == g1[name]).all(), name


def test_route_ex_with_reroute_matches_forward_ex():
    cfg = MoEConfig("bf16_reroute_route", 1500, 128, 32, 2, 128, 1.0, "bf16", seed=50,
                    zipf_bias=True)
    inp = inputs.make_separated_inputs(cfg)
    g, (c, dev, ws, opts) = run_opts(cfg, inp, reroute=True)
    r = moe.route(c, dev.x, dev.w_router, dev.router_bias, workspace=ws,
                  options=moe.Options(reroute=True))
    assert moe.get_status(ws) == 0
    for name in ("topk_idx", "topk_w", "aux_loss", "drop_mask", "expert_counts", "kept_counts"):
        assert (getattr(r, name).cpu().numpy() == g[name]).all(), name


# ------------------------------------- overflow rerouting on ordinary router logits
#
# Inputs from the ordinary recipe (inputs.make_inputs): the GPU's fp32 logits differ
# from the oracle's fp64 ones by accumulation rounding, so near ties may resolve
# differently. The comparison conditions on the GPU's own routing before rerouting
# (the same call without the option), as the capacity comparison above does:
#
# 1. that routing must match the oracle's, except tokens in its near-tie set (set
#    flips) or near-tie order set (slot order);
# 2. a conditional oracle runs capacity and one round of rerouting on it with the
#    fp64 logits (oracle.capacity_assign, oracle.reroute_overflow);
# 3. a token whose dropped slots' proposals may flip (oracle.reroute_near_ties) can
#    change which proposals reach which expert, so the experts in its tied groups
#    are "affected". Every token that is not tied and proposes no affected expert
#    must match the conditional oracle exactly; the others must be a valid outcome
#    (distinct experts, moves only from dropped slots to experts with room that the
#    token did not select, among its first m+1 candidates, room respected);
# 4. outputs: the oracle's expert FFNs and combine (oracle.experts_combine) on the
#    GPU's final routing with the fp64 gate weights of the GPU's first routing.

def _candidates(logits_t, own, counts, C):
    """Experts a token may move to, best first (brute force)."""
    return sorted((e for e in range(len(logits_t)) if counts[e] < C and e not in own),
                  key=lambda e: (-logits_t[e], e))


def check_reroute_ordinary(cfg, token_sample=None, want_split=None):
    inp = inputs.make_inputs(cfg)
    g, (c, dev, ws, opts) = run_opts(cfg, inp, reroute=True)
    if want_split is not None:
        assert (moe.describe(c)["router_ksplit"] > 1) == want_split
    r0 = moe.route(c, dev.x, dev.w_router, dev.router_bias)   # the routing before rerouting
    idx0 = r0.topk_idx.cpu().numpy().astype(np.int64)
    w0 = r0.topk_w.cpu().numpy()
    drop0_g = r0.drop_mask.cpu().numpy()
    T, k, N = cfg.T, cfg.k, cfg.N
    x, wr = inp.values("x"), inp.values("w_router")
    ref = orc.route(x, wr, inp.router_bias, k, cfg.capacity_factor)
    L = ref["logits"]
    C = ref["capacity"]

    # 1. the first routing against the oracle's
    same_set = (np.sort(idx0, axis=1) == np.sort(ref["topk_idx"], axis=1)).all(axis=1)
    flipped = np.nonzero(~same_set)[0]
    assert set(flipped.tolist()) <= set(ref["near_tie_set"].tolist())
    reordered = np.nonzero(same_set & (idx0 != ref["topk_idx"]).any(axis=1))[0]
    assert set(reordered.tolist()) <= set(ref["near_tie_order"].tolist())
    w_ref = orc.gate_weights(L, idx0)
    assert np.abs(w0 - w_ref).max() <= TOL_W
    assert abs(float(g["aux_loss"][0]) - ref["aux_loss"]) <= TOL_AUX

    # 2. the conditional oracle on the GPU's first routing
    counts = orc.expert_counts(idx0, N)
    _, drop0, _ = orc.capacity_assign(idx0, N, C)
    assert (drop0_g == drop0).all()
    assert (g["expert_counts"] == counts).all()           # the original routing's counts
    idx_c, drop_c, rer_c, acc_c = orc.reroute_overflow(L, idx0, drop0, counts, C)
    ties = set(orc.reroute_near_ties(L, idx0, drop0, counts, C).tolist())

    # 3. affected experts: the tied groups among each tied token's first m+1
    #    candidates, each from the first tied token that may propose it (experts
    #    accept in token order, so earlier proposals are not affected)
    first_tie = {}
    props = {}
    for t in np.nonzero(drop0.any(axis=1))[0]:
        m = int(drop0[t].sum())
        cand = _candidates(L[t], set(idx0[t].tolist()), counts, C)
        props[t] = cand[:m]
        if t in ties:
            v = L[t][cand[:m + 1]]
            for j in range(len(v) - 1):
                if v[j] - v[j + 1] < orc.NEAR_TIE_MARGIN:
                    for e in (cand[j], cand[j + 1]):
                        first_tie.setdefault(e, t)
    affected = set(first_tie)
    idx_f, drop_f = g["topk_idx"].astype(np.int64), g["drop_mask"]
    exact = np.array([t not in ties and all(t < first_tie.get(e, T) for e in props.get(t, []))
                      for t in range(T)])
    assert (idx_f[exact] == idx_c[exact]).all(), "final experts differ"
    assert (drop_f[exact] == drop_c[exact]).all(), "final drops differ"
    assert (g["topk_w"] == w0).all()                       # moved slots keep their weights
    moved = idx_f != idx0
    assert (drop0[moved] == 1).all() and (drop_f[moved] == 0).all()
    room = np.maximum(C - counts, 0)
    for t in np.nonzero(~exact)[0]:
        assert len(set(idx_f[t].tolist())) == k
        m = int(drop0[t].sum())
        cand = _candidates(L[t], set(idx0[t].tolist()), counts, C)[:m + 1]
        for s in np.nonzero(moved[t])[0]:
            assert idx_f[t, s] in cand
    final = np.bincount(idx_f[drop_f == 0], minlength=N)
    assert (g["kept_counts"] == final).all() and (final <= C).all()
    assert (np.bincount(idx_f[moved], minlength=N) <= room).all()

    # 4. outputs on the GPU's final routing
    tokens = np.arange(T) if token_sample is None else np.asarray(token_sample)
    y_ref = orc.experts_combine(x, inp.values("w1"), inp.values("w3"), inp.values("w2"),
                                idx_f, w_ref, drop_f, tokens)
    dead = drop_f[tokens].all(axis=1)
    assert (g["out"][tokens[dead]] == 0).all()
    err = _rel_err(g["out"][tokens[~dead]], y_ref[~dead])
    info = dict(err=err, max_ratio=_max_ratio(g["out"][tokens[~dead]], y_ref[~dead]),
                near_tie_set=len(ref["near_tie_set"]),
                near_tie_order=len(ref["near_tie_order"]), flipped=len(flipped),
                reroute_ties=len(ties), affected_experts=len(affected),
                checked_exactly=int(exact.sum()), rerouted=int(moved.sum()),
                dropped=int(drop_f.sum()))
    parity_report.record(f"{cfg.name} (ordinary logits, rerouting)", **info)
    assert err <= TOL[cfg.dtype], f"output relative error {err:.3e} > {TOL[cfg.dtype]}"
    assert info["rerouted"] > 0
    return info


REROUTE_ORDINARY = [
    # the fused routing kernel (>= 32 tiles of 128 tokens), Zipf-skewed experts
    (MoEConfig("bf16_reroute_real_fused_zipf", 4096, 256, 32, 2, 128, 1.1, "bf16", seed=61,
               zipf_bias=True), False),
    # the split-K tensor-core router and the routing-decision kernel
    (MoEConfig("bf16_reroute_real_splitk", 1500, 512, 16, 2, 256, 0.9, "bf16", seed=62,
               zipf_bias=True), True),
    # float32: CUDA-core router
    (MoEConfig("f32_reroute_real", 300, 192, 16, 2, 320, 1.0, "f32", seed=63, zipf_bias=True),
     None),
    # k = 4 with hot and cold experts (a uniform router at CF < 1 would leave no room)
    (MoEConfig("bf16_reroute_real_k4", 2000, 256, 16, 4, 128, 1.0, "bf16", seed=64,
               zipf_bias=True), None),
]


@pytest.mark.parametrize("case", REROUTE_ORDINARY, ids=lambda c: c[0].name)
def test_reroute_on_ordinary_logits(case):
    cfg, split = case
    check_reroute_ordinary(cfg, want_split=split)


def test_reroute_on_the_finegrained_workload_sampled():
    # the fine-grained Zipf-skewed workload itself: routing for every token, outputs on
    # a seeded sample of rows
    cfg = configs.FINEGRAINED_T16384
    sample = np.sort(np.random.default_rng(11).choice(cfg.T, size=256, replace=False))
    check_reroute_ordinary(cfg, token_sample=sample)
