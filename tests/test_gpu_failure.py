"""Failure detection on the GPU without a fault: a device-side bounded wait that runs
out.

The test build of the library (libmoe_b300_testhooks.so, include/moe_test_hooks.h)
can have the bf16 expert GEMM on single-CTA tiles withhold the TMA loads of one
k-chunk in its first CTA. That stage's barrier then never completes: the MMA thread's
bounded wait (2 s) gives up, sets status bit 1 and the abort flag, the producer lets
the loads it did issue land, the MMA thread waits for the MMAs it did issue, the
epilogue leaves on the abort flag, tensor memory is freed and the kernel returns.
The host reads MOE_EDEVICE with bit 1 from moe_get_status; the next call on the same
workspace, with nothing withheld, must succeed and match the oracle.
"""
import ctypes

import pytest
import torch

import oracle as orc
from mixture_experts_layer_102_b300 import build, inputs, moe
from mixture_experts_layer_102_b300.configs import MoEConfig

pytestmark = pytest.mark.gpu

# 300 tokens over 8 experts: ~75 rows per expert, 128-row tiles on single CTAs; K = 128
# for GEMM1, so k-chunk 1 (the second of two) is withheld after chunk 0 was consumed.
CFG = MoEConfig("bf16_wait_gives_up", 300, 128, 8, 2, 128, None, "bf16", seed=70)


@pytest.fixture()
def hooks_lib(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = build.build_test_hooks(quiet=True)
    lib = ctypes.CDLL(path)
    for name, (res, args) in moe._SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    lib.moe_test_withhold_gemm_load.restype = None
    lib.moe_test_withhold_gemm_load.argtypes = [ctypes.c_int]
    monkeypatch.setattr(moe, "_lib", lib)   # the binding calls the test build
    yield lib
    lib.moe_test_withhold_gemm_load(-1)


def test_bounded_wait_gives_up_and_the_next_call_recovers(hooks_lib):
    import test_gpu_parity as parity
    assert moe.describe(moe.cfg_from(CFG))["gemm1_tile_rows"] == 128
    inp = inputs.make_inputs(CFG)
    dev = moe.to_device(inp)
    c = moe.cfg_from(CFG)
    ws = moe.make_workspace(c)
    routing = moe.new_routing(c)
    stream = torch.cuda.current_stream()

    hooks_lib.moe_test_withhold_gemm_load(1)
    moe.forward(c, dev.x, dev.w_router, dev.router_bias, dev.w1, dev.w3, dev.w2,
                workspace=ws, routing=routing)
    bits = ctypes.c_uint32(0)
    rc = hooks_lib.moe_get_status(ws.data_ptr(), ws.numel(), stream.cuda_stream,
                                  ctypes.byref(bits))
    assert rc == moe.MOE_EDEVICE and (bits.value & 1), (rc, bits.value)

    hooks_lib.moe_test_withhold_gemm_load(-1)
    out = moe.forward(c, dev.x, dev.w_router, dev.router_bias, dev.w1, dev.w3, dev.w2,
                      workspace=ws, routing=routing)
    assert moe.get_status(ws) == 0       # the status word was cleared by the read above
    g = {k: getattr(routing, k).cpu().numpy() for k in
         ("topk_idx", "topk_w", "aux_loss", "drop_mask", "expert_counts", "kept_counts")}
    g["out"] = out.float().cpu().numpy()
    ref = orc.moe_forward(inp.values("x"), inp.values("w_router"), inp.router_bias,
                          inp.values("w1"), inp.values("w3"), inp.values("w2"), CFG.k,
                          CFG.capacity_factor)
    parity.compare(CFG, g, ref)
