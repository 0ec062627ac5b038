"""Host-side checks of the C-ABI library: it loads, exports every function that
include/moe.h declares, and its pure-host logic (workspace sizing, capacity, argument
validation) behaves as documented. No call here reaches a CUDA launch: every failing
argument check returns before the library touches the CUDA API."""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import oracle as orc
from mixture_experts_layer_102_b300 import build, configs, inputs, moe

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build(quiet=True)


def _declared_functions():
    text = (ROOT / "include" / "moe.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = _declared_functions()
    assert set(names) == set(moe._SIGNATURES), names
    lib = moe.library()
    for name in names:
        assert getattr(lib, name) is not None


def test_strerror_covers_every_status():
    for code in range(8):
        assert moe.strerror(code) != "unknown status"
    assert moe.strerror(99) == "unknown status"


@pytest.mark.parametrize("c", configs.NAMED, ids=lambda c: c.name)
def test_workspace_size_positive_and_linear_in_tokens(c):
    s1 = moe.workspace_size(moe.cfg_from(c))
    s2 = moe.workspace_size(moe.cfg_from(c, T=2 * c.T))
    assert s1 > 0 and s2 > s1
    elem = 2 if c.dtype == "bf16" else 4
    # the permuted rows, h and ye dominate: at least T*k*(2H+F) elements when no
    # capacity limit bounds them
    if c.capacity_factor is None:
        assert s1 >= c.T * c.k * (2 * c.H + c.F) * elem


def test_workspace_size_zero_for_invalid():
    lib = moe.library()
    bad = [moe.make_cfg(64, 100, 8, 2, 256, None, "bf16"),     # H % 64
           moe.make_cfg(64, 128, 8, 9, 256, None, "bf16"),     # k > N
           moe.make_cfg(64, 128, 300, 2, 256, None, "bf16"),   # N > 256
           moe.make_cfg(-1, 128, 8, 2, 256, None, "bf16")]
    for cfg in bad:
        assert lib.moe_workspace_size(ctypes.byref(cfg)) == 0
    assert lib.moe_workspace_size(None) == 0


def test_capacity_matches_oracle():
    rng = np.random.default_rng(0)
    for c in configs.NAMED:
        assert moe.capacity(moe.cfg_from(c)) == orc.capacity(c.T, c.k, c.N, c.capacity_factor)
    for _ in range(500):
        T = int(rng.integers(1, 50000))
        N = int(rng.integers(1, 257))
        k = int(rng.integers(1, min(N, 32) + 1))
        cf = float(np.float32(rng.uniform(0.01, 3.0)))
        got = moe.capacity(moe.make_cfg(T, 64, N, k, 64, cf, "bf16"))
        want = orc.capacity(T, k, N, cf)
        assert got == min(want, T * k)
    assert moe.capacity(moe.make_cfg(10, 64, 4, 2, 64, None, "f32")) is None


def _args(cfg, **over):
    """Plausible fake device pointers; the calls below fail validation first."""
    d = dict(x=0x10000, wr=0x20000, bias=None, w1=0x30000, w3=0x40000, w2=0x50000,
             out=0x60000, ws=0x100000, ws_bytes=moe.workspace_size(cfg))
    d.update(over)
    return d


def _forward(cfg, a):
    return moe.library().moe_forward(ctypes.byref(cfg), a["x"], a["wr"], a["bias"], a["w1"],
                                     a["w3"], a["w2"], a["out"], None, None, None, None, None,
                                     None, a["ws"], a["ws_bytes"], None)


def test_forward_rejects_bad_arguments_before_any_cuda_call():
    cfg = moe.cfg_from(configs.BF16_T4096)
    assert _forward(cfg, _args(cfg, x=None)) == moe.MOE_EINVAL
    assert _forward(cfg, _args(cfg, w2=None)) == moe.MOE_EINVAL
    assert _forward(cfg, _args(cfg, out=0x60008)) == moe.MOE_EALIGN
    assert _forward(cfg, _args(cfg, bias=0x7002)) == moe.MOE_EALIGN
    assert _forward(cfg, _args(cfg, ws=None)) == moe.MOE_EWORKSPACE
    assert _forward(cfg, _args(cfg, ws=0x100010)) == moe.MOE_EWORKSPACE
    a = _args(cfg)
    a["ws_bytes"] -= 1
    assert _forward(cfg, a) == moe.MOE_EWORKSPACE
    bad_h = moe.make_cfg(64, 96, 8, 2, 256, None, "bf16")
    assert _forward(bad_h, _args(cfg)) == moe.MOE_EUNSUPPORTED
    bad_k = moe.make_cfg(64, 128, 4, 5, 256, None, "bf16")
    assert _forward(bad_k, _args(cfg)) == moe.MOE_EINVAL
    bad_dtype = moe.make_cfg(64, 128, 4, 2, 256, None, "bf16")
    bad_dtype.dtype = 7
    assert _forward(bad_dtype, _args(cfg)) == moe.MOE_EINVAL


def test_route_requires_its_outputs():
    cfg = moe.cfg_from(configs.TINY_F32)
    lib = moe.library()
    ws_bytes = moe.workspace_size(cfg)
    rc = lib.moe_route(ctypes.byref(cfg), 0x10000, 0x20000, None, None, 0x30000, 0x40000,
                       0x50000, None, None, 0x100000, ws_bytes, None)
    assert rc == moe.MOE_EINVAL
    rc = lib.moe_route(ctypes.byref(cfg), 0x10000, 0x20000, None, 0x30002, 0x30000, 0x40000,
                       0x50000, None, None, 0x100000, ws_bytes, None)
    assert rc == moe.MOE_EALIGN


def test_status_and_init_reject_bad_workspace():
    lib = moe.library()
    assert lib.moe_workspace_init(None, 1024, None) == moe.MOE_EWORKSPACE
    assert lib.moe_workspace_init(0x100001, 1024, None) == moe.MOE_EWORKSPACE
    assert lib.moe_get_status(0x100000, 16, None, None) == moe.MOE_EWORKSPACE


def test_binding_checks_shapes_without_a_gpu():
    import torch
    cfg = moe.cfg_from(configs.TINY_F32)
    x = torch.zeros(cfg.T, cfg.H)
    with pytest.raises(ValueError):
        moe.route(cfg, x, torch.zeros(cfg.H, cfg.N))   # CPU tensors are refused


def _opts(n_shared=0, activation=moe.MOE_ACT_SWIGLU, valid=None):
    return moe.MoEOptions(n_shared, activation, valid, None, None)


def test_workspace_size_ex_matches_base_and_grows_with_shared_experts():
    lib = moe.library()
    for c in configs.NAMED:
        cfg = moe.cfg_from(c)
        base = moe.workspace_size(cfg)
        assert lib.moe_workspace_size_ex(ctypes.byref(cfg), None) == base
        assert lib.moe_workspace_size_ex(ctypes.byref(cfg), ctypes.byref(_opts())) == base
        s2 = lib.moe_workspace_size_ex(ctypes.byref(cfg), ctypes.byref(_opts(2)))
        elem = 2 if c.dtype == "bf16" else 4
        # two more rows per token in the permuted input, h and the expert outputs
        assert s2 >= base + 2 * c.T * (2 * c.H + c.F) * elem


def test_workspace_size_ex_zero_for_bad_options():
    lib = moe.library()
    cfg = moe.cfg_from(configs.TINY_F32)
    for o in (_opts(-1), _opts(moe.MOE_MAX_SHARED + 1), _opts(0, 2), _opts(0, -1)):
        assert lib.moe_workspace_size_ex(ctypes.byref(cfg), ctypes.byref(o)) == 0
    assert lib.moe_workspace_size_ex(ctypes.byref(cfg), ctypes.byref(_opts(8))) > 0


def test_ex_calls_reject_bad_options_before_any_cuda_call():
    lib = moe.library()
    cfg = moe.cfg_from(configs.BF16_T4096)
    a = _args(cfg)
    fwd = lambda o, w3=a["w3"]: lib.moe_forward_ex(
        ctypes.byref(cfg), ctypes.byref(o), a["x"], a["wr"], a["bias"], a["w1"], w3, a["w2"],
        a["out"], None, None, None, None, None, None, a["ws"], a["ws_bytes"], None, None)
    assert fwd(_opts(9)) == moe.MOE_EINVAL
    assert fwd(_opts(0, 5)) == moe.MOE_EINVAL
    assert fwd(_opts(0, moe.MOE_ACT_SWIGLU), w3=None) == moe.MOE_EINVAL   # SwiGLU needs W3
    bad_kl = moe.MoEOptions(0, 0, None, 0x7002, None)
    assert fwd(bad_kl) == moe.MOE_EALIGN
    rc = lib.moe_route_ex(ctypes.byref(cfg), ctypes.byref(_opts(-3)), a["x"], a["wr"], None,
                          0x30000, 0x40000, 0x50000, 0x60000, None, None, a["ws"],
                          a["ws_bytes"], None)
    assert rc == moe.MOE_EINVAL
    # the base workspace is too small once shared experts add rows
    assert fwd(_opts(1)) == moe.MOE_EWORKSPACE


def test_options_binding_checks_without_a_gpu():
    import torch
    with pytest.raises(ValueError):
        moe.Options(activation="relu").to_c()
    with pytest.raises(ValueError):
        moe.Options(valid_mask=torch.ones(4, dtype=torch.uint8)).check(4)   # CPU tensor


def _plan(config, options=None, has_bias=False, **over):
    cfg = config.with_(**over) if over else config
    return moe.describe(moe.cfg_from(cfg), options, has_bias)


def test_describe_reports_the_plan_of_each_workload():
    # the bench layer: fused routing on 128-token blocks, GEMM1 on CTA pairs (512 rows
    # per expert, 256-row tiles compute at most 12% more rows), GEMM2 on single CTAs
    p = _plan(configs.BF16_T4096)
    assert (p["fused_routing"], p["routing_block"], p["router_ksplit"]) == (1, 128, 1)
    assert (p["gemm1_tile_rows"], p["gemm2_tile_rows"]) == (256, 128)
    assert p["launches"] == 5 and p["capacity"] == 640
    assert p["workspace_bytes"] == moe.workspace_size(moe.cfg_from(configs.BF16_T4096))
    # with a router bias GEMM1 keeps the 1024-rows-per-expert rule for pairs
    assert _plan(configs.BF16_T4096, has_bias=True)["gemm1_tile_rows"] == 128
    # Mixtral-shaped: 2048 rows per expert, both GEMMs on pairs
    p = _plan(configs.MIXTRAL_T8192)
    assert (p["fused_routing"], p["gemm1_tile_rows"], p["gemm2_tile_rows"]) == (1, 256, 256)
    assert p["capacity"] == 3072
    # fine-grained with its Zipf bias: 512 rows per expert, single CTAs for both
    p = _plan(configs.FINEGRAINED_T16384, has_bias=True)
    assert (p["fused_routing"], p["gemm1_tile_rows"], p["gemm2_tile_rows"]) == (1, 128, 128)
    assert p["capacity"] == 615
    # decode: one tile of tokens, so the router splits K and the decisions follow
    p = _plan(configs.DECODE_T64)
    assert p["fused_routing"] == 0 and p["router_ksplit"] > 1 and p["launches"] == 6
    assert p["capacity"] == -1 and (p["gemm1_tile_rows"], p["gemm2_tile_rows"]) == (128, 128)
    # float32: the SIMT path, never fused
    p = _plan(configs.TINY_F32)
    assert p["fused_routing"] == 0 and p["launches"] == 6


def test_describe_fused_threshold_and_options():
    # fused from 32 tiles of 128 tokens on: T = 3968 is 31 tiles, T = 3969 is 32
    assert _plan(configs.BF16_T4096, T=3968)["fused_routing"] == 0
    assert _plan(configs.BF16_T4096, T=3969)["fused_routing"] == 1
    assert _plan(configs.BF16_T4096, T=3969, dtype="f32")["fused_routing"] == 0
    # rerouting adds a launch when there is a capacity limit, and nothing without one
    rr = moe.Options(reroute=True)
    assert _plan(configs.BF16_T4096, rr)["launches"] == 6
    assert _plan(configs.BF16_T4096, rr, capacity_factor=None)["launches"] == 5
    # shared experts count as experts of T rows each in the tile choice and workspace
    sh = moe.Options(n_shared=2)
    c = moe.cfg_from(configs.BF16_T4096)
    assert _plan(configs.BF16_T4096, sh)["workspace_bytes"] == moe.workspace_size(c, sh)


def test_describe_routing_finish_and_threads():
    import torch
    fin = lambda p: (p["routing_threads"], p["routing_warp_finish"])
    # fused kernel: one-warp finish while 32/np2(N) lanes x 16 rows cover the blocks
    assert fin(_plan(configs.BF16_T4096)) == (256, 1)            # N 16: 2 lanes, 32 blocks
    assert fin(_plan(configs.BF16_T4096, T=4097)) == (256, 0)    # 33 blocks
    assert fin(_plan(configs.MIXTRAL_T8192)) == (256, 1)         # N 8: 4 lanes, 64 blocks
    assert fin(_plan(configs.MIXTRAL_T8192, T=8193)) == (256, 0)
    assert fin(_plan(configs.BF16_T4096, N=17)) == (256, 0)      # np2 32: one lane, 16 rows
    # above 32 experts the fused kernel runs four threads per token and the block finish
    assert fin(_plan(configs.FINEGRAINED_T16384)) == (512, 0)
    assert fin(_plan(configs.BF16_T4096, N=33)) == (512, 0)
    # the routing-decision kernel (1024 threads): 8 rows per lane, any N
    assert fin(_plan(configs.DECODE_T64)) == (1024, 1)           # N 100: 2 blocks
    assert fin(_plan(configs.BF16_T4096, T=200, N=256, k=4)) == (1024, 1)   # 7 blocks
    assert fin(_plan(configs.BF16_T4096, T=257, N=256, k=4)) == (1024, 0)   # 9 blocks
    assert fin(_plan(configs.TINY_F32)) == (1024, 1)
    # a mask or an optional loss keeps the block finish
    one = torch.zeros(1, dtype=torch.float32)
    mask = torch.ones(configs.BF16_T4096.T, dtype=torch.uint8)
    for o in (moe.Options(aux_kl=one), moe.Options(aux_std2=one), moe.Options(valid_mask=mask)):
        assert fin(_plan(configs.BF16_T4096, o)) == (256, 0)
        assert fin(_plan(configs.DECODE_T64, o))[1] == 0
    # shared experts and rerouting do not change the choice
    assert fin(_plan(configs.BF16_T4096, moe.Options(n_shared=2, reroute=True))) == (256, 1)


def test_describe_rejects_bad_arguments():
    lib = moe.library()
    plan = moe.MoEPlan()
    c = moe.cfg_from(configs.BF16_T4096)
    assert lib.moe_describe(ctypes.byref(c), None, 0, None) == moe.MOE_EINVAL
    assert lib.moe_describe(None, None, 0, ctypes.byref(plan)) == moe.MOE_EINVAL
    bad = moe.make_cfg(T=64, H=128, N=4, k=5, F=64, capacity_factor=None, dtype="bf16")
    assert lib.moe_describe(ctypes.byref(bad), None, 0, ctypes.byref(plan)) == moe.MOE_EINVAL
    big = moe.make_cfg(T=64, H=128, N=300, k=2, F=64, capacity_factor=None, dtype="bf16")
    assert lib.moe_describe(ctypes.byref(big), None, 0, ctypes.byref(plan)) == \
        moe.MOE_EUNSUPPORTED
    with pytest.raises(moe.MoEError):
        moe.describe(c, moe.Options(n_shared=99))


@pytest.mark.parametrize("config,has_bias", [(configs.BF16_T4096, False),
                                             (configs.MIXTRAL_T8192, False),
                                             (configs.FINEGRAINED_T16384, True)])
def test_gemm1_tile_choice_agrees_with_the_padding_of_real_routing(config, has_bias):
    # the host picks 256-row pair tiles for GEMM1 from a model of the expert counts; on
    # the seeded workloads the oracle's kept counts must bear the choice out: pairs only
    # where 256-row tiles compute at most 12% more rows than 128-row tiles
    inp = inputs.make_inputs(config, with_experts=False)
    r = orc.route(inp.values("x"), inp.values("w_router"), inp.router_bias, config.k,
                  config.capacity_factor)
    kept = r["kept_counts"]
    rows = {m: int(sum(-(-int(c) // m) * m for c in kept)) for m in (128, 256)}
    ratio = rows[256] / rows[128]
    pair = moe.describe(moe.cfg_from(config), has_bias=has_bias)["gemm1_tile_rows"] == 256
    assert pair == (ratio <= 1.12), (config.name, rows, ratio)
