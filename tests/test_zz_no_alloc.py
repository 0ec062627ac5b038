"""moe_route_static: routing for callers that cannot allocate device memory (plugin
hosts and serving runtimes that plan every device buffer themselves and do not let
a kernel library call cudaMalloc). Its scratch is a static device array inside the
library; these tests check that it gives the same routing as moe_route, which uses a
caller-provided workspace, on two calls in a row (the array keeps the previous
call's contents), that moe_get_status_static finds no failure reported after each
call, and that a layer too large for the array is refused on the host.

This file is collected last so that a failure here, in a run that stops at the first
failure, comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_102_b300 import configs, inputs, moe
from mixture_experts_layer_102_b300.configs import MoEConfig

TOL_W = 1e-5     # gate weights, as in the parity tests
TOL_AUX = 1e-5   # aux loss, as in the parity tests


def _status_static():
    bits = ctypes.c_uint32(0xFFFFFFFF)
    rc = moe.library().moe_get_status_static(torch.cuda.current_stream().cuda_stream,
                                             ctypes.byref(bits))
    return rc, bits.value


def _route_static(c, dev, r):
    lib = moe.library()
    p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return lib.moe_route_static(ctypes.byref(c), p(dev.x), p(dev.w_router), p(dev.router_bias),
                                p(r.topk_idx), p(r.topk_w), p(r.aux_loss), p(r.drop_mask),
                                p(r.expert_counts), p(r.kept_counts),
                                torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [
    configs.BF16_T4096,
    MoEConfig("bf16_zipf_drops_static", 3000, 256, 64, 2, 128, 1.2, "bf16", seed=11,
              zipf_bias=True),
    configs.TINY_F32,
], ids=lambda c: c.name)
def test_static_route_matches_workspace_route(cfg):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_102_b300 import build
    build.build(quiet=True)
    inp = inputs.make_inputs(cfg, with_experts=False)
    dev = moe.to_device(inp)
    c = moe.cfg_from(cfg)
    ref = moe.route(c, dev.x, dev.w_router, dev.router_bias)
    torch.cuda.synchronize()
    for _ in range(2):
        got = moe.new_routing(c)
        assert _route_static(c, dev, got) == moe.MOE_OK
        assert _status_static() == (moe.MOE_OK, 0)   # no kernel reported a failure
        assert (got.topk_idx == ref.topk_idx).all()
        assert (got.topk_w - ref.topk_w).abs().max().item() <= TOL_W
        assert abs(got.aux_loss.item() - ref.aux_loss.item()) <= TOL_AUX
        assert (got.drop_mask == ref.drop_mask).all()
        assert (got.expert_counts == ref.expert_counts).all()
        assert (got.kept_counts == ref.kept_counts).all()


def test_static_route_refuses_a_layer_beyond_the_scratch_size():
    # 256 experts x 65536 tokens needs 64 MiB of partial logits alone: refused before
    # any CUDA call (the pointers below are never dereferenced).
    c = moe.make_cfg(65536, 1024, 256, 2, 1024, 1.0, "bf16")
    lib = moe.library()
    rc = lib.moe_route_static(ctypes.byref(c), 0x10000, 0x20000, None, 0x30000, 0x40000,
                              0x50000, 0x60000, None, None, None)
    assert rc == moe.MOE_EUNSUPPORTED
