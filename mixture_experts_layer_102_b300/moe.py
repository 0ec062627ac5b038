"""Python binding of the C-ABI library ``libmoe_b300.so`` (include/moe.h).

Argument marshalling only: the functions check dtypes, devices and shapes, allocate
output tensors with torch on the caller's behalf and pass raw device pointers to
the library. Every step of the layer runs in the library's CUDA kernels. There is
no CPU path: on a machine without the library or without an sm_103 GPU the calls
raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK, MOE_EINVAL, MOE_EUNSUPPORTED, MOE_EWORKSPACE, MOE_EALIGN = 0, 1, 2, 3, 4
MOE_ECUDA, MOE_EDEVICE, MOE_ENODEVICE = 5, 6, 7
MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_SWIGLU, MOE_ACT_GELU = 0, 1
MOE_MAX_SHARED = 8
MOE_NUM_STAGES = 6
STAGE_NAMES = ["router_logits", "route_select", "dispatch", "gemm1_swiglu", "gemm2", "combine"]

# Every function the header declares, with its C signature.
_P = ctypes.c_void_p
_SIGNATURES = {
    "moe_workspace_size": (ctypes.c_size_t, [_P]),
    "moe_capacity": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int64)]),
    "moe_workspace_init": (ctypes.c_int, [_P, ctypes.c_size_t, _P]),
    "moe_route": (ctypes.c_int, [_P] + [_P] * 9 + [_P, ctypes.c_size_t, _P]),
    "moe_forward": (ctypes.c_int, [_P] + [_P] * 13 + [_P, ctypes.c_size_t, _P]),
    "moe_forward_timed": (ctypes.c_int, [_P] + [_P] * 13 + [_P, ctypes.c_size_t, _P, _P]),
    "moe_get_status": (ctypes.c_int, [_P, ctypes.c_size_t, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_route_static": (ctypes.c_int, [_P] + [_P] * 9 + [_P]),
    "moe_get_status_static": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_workspace_size_ex": (ctypes.c_size_t, [_P, _P]),
    "moe_describe": (ctypes.c_int, [_P, _P, ctypes.c_int, _P]),
    "moe_route_ex": (ctypes.c_int, [_P, _P] + [_P] * 9 + [_P, ctypes.c_size_t, _P]),
    "moe_forward_ex": (ctypes.c_int, [_P, _P] + [_P] * 13 + [_P, ctypes.c_size_t, _P, _P]),
    "moe_strerror": (ctypes.c_char_p, [ctypes.c_int]),
}


class MoECfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32),
                ("k", ctypes.c_int32), ("F", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("dtype", ctypes.c_int32)]


class MoEOptions(ctypes.Structure):
    _fields_ = [("n_shared", ctypes.c_int32), ("activation", ctypes.c_int32),
                ("valid_mask", ctypes.c_void_p), ("aux_kl", ctypes.c_void_p),
                ("aux_std2", ctypes.c_void_p), ("reroute", ctypes.c_int32)]


@dataclass
class Options:
    """The layer variants of moe_options: shared experts, the GELU expert, a
    valid-token mask ([T] uint8 or bool on the device), the two extra balance
    losses (pass [1] float32 device tensors to receive them) and overflow rerouting."""
    n_shared: int = 0
    activation: str = "swiglu"
    valid_mask: Optional[torch.Tensor] = None
    aux_kl: Optional[torch.Tensor] = None
    aux_std2: Optional[torch.Tensor] = None
    reroute: bool = False

    def to_c(self) -> MoEOptions:
        if self.activation not in ("swiglu", "gelu"):
            raise ValueError(f"activation must be 'swiglu' or 'gelu', got {self.activation!r}")
        return MoEOptions(int(self.n_shared),
                          MOE_ACT_GELU if self.activation == "gelu" else MOE_ACT_SWIGLU,
                          _ptr(self.valid_mask), _ptr(self.aux_kl), _ptr(self.aux_std2),
                          1 if self.reroute else 0)

    def check(self, T: int):
        if self.valid_mask is not None:
            if self.valid_mask.dtype not in (torch.uint8, torch.bool):
                raise ValueError("valid_mask must be uint8 or bool")
            if not self.valid_mask.is_cuda or tuple(self.valid_mask.shape) != (T,) \
                    or not self.valid_mask.is_contiguous():
                raise ValueError(f"valid_mask must be a contiguous CUDA tensor of shape ({T},)")
        for name in ("aux_kl", "aux_std2"):
            t = getattr(self, name)
            if t is not None:
                _check(t, name, (1,), torch.float32)


class MoEPlan(ctypes.Structure):
    _fields_ = [("fused_routing", ctypes.c_int32), ("routing_block", ctypes.c_int32),
                ("router_ksplit", ctypes.c_int32), ("gemm1_tile_rows", ctypes.c_int32),
                ("gemm2_tile_rows", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("capacity", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("routing_threads", ctypes.c_int32), ("routing_warp_finish", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({strerror(status)})")
        self.status = status


_lib = None


def library() -> ctypes.CDLL:
    """Load the shared library (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mixture_experts_layer_102_b300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def strerror(status: int) -> str:
    return library().moe_strerror(int(status)).decode()


def make_cfg(T: int, H: int, N: int, k: int, F: int, capacity_factor: Optional[float],
             dtype: str) -> MoECfg:
    cf = 0.0 if capacity_factor is None else float(capacity_factor)
    return MoECfg(int(T), int(H), int(N), int(k), int(F), cf,
                  MOE_BF16 if dtype == "bf16" else MOE_F32)


def cfg_from(config, T: Optional[int] = None) -> MoECfg:
    """MoECfg of a configs.MoEConfig (optionally with another token count)."""
    return make_cfg(config.T if T is None else T, config.H, config.N, config.k, config.F,
                    config.capacity_factor, config.dtype)


def workspace_size(cfg: MoECfg, options: Optional[Options] = None) -> int:
    if options is None:
        n = library().moe_workspace_size(ctypes.byref(cfg))
    else:
        n = library().moe_workspace_size_ex(ctypes.byref(cfg), ctypes.byref(options.to_c()))
    if n == 0:
        raise MoEError("moe_workspace_size", MOE_EINVAL)
    return int(n)


def describe(cfg: MoECfg, options: Optional[Options] = None, has_bias: bool = False) -> dict:
    """moe_describe: the plan moe_forward follows for cfg (host only, no GPU needed)."""
    plan = MoEPlan()
    opts = None if options is None else ctypes.byref(options.to_c())
    rc = library().moe_describe(ctypes.byref(cfg), opts, 1 if has_bias else 0,
                                ctypes.byref(plan))
    if rc != MOE_OK:
        raise MoEError("moe_describe", rc)
    return {name: getattr(plan, name) for name, _ in MoEPlan._fields_}


def capacity(cfg: MoECfg) -> Optional[int]:
    c = ctypes.c_int64(0)
    rc = library().moe_capacity(ctypes.byref(cfg), ctypes.byref(c))
    if rc != MOE_OK:
        raise MoEError("moe_capacity", rc)
    return None if c.value < 0 else int(c.value)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def make_workspace(cfg: MoECfg, device=None, options: Optional[Options] = None) -> torch.Tensor:
    """A zeroed device workspace for `cfg` (the library allocates nothing itself)."""
    n = workspace_size(cfg, options)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _io_dtype(cfg: MoECfg) -> torch.dtype:
    return torch.bfloat16 if cfg.dtype == MOE_BF16 else torch.float32


def _check(t: torch.Tensor, name: str, shape: Sequence[int], dtype: torch.dtype):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


@dataclass
class Routing:
    topk_idx: torch.Tensor       # [T,k] int32
    topk_w: torch.Tensor         # [T,k] float32
    aux_loss: torch.Tensor       # [1] float32
    drop_mask: torch.Tensor      # [T,k] uint8
    expert_counts: torch.Tensor  # [N] int32
    kept_counts: torch.Tensor    # [N] int32


def _routing_outputs(cfg: MoECfg, device) -> Routing:
    T, k, N = cfg.T, cfg.k, cfg.N
    return Routing(torch.empty((T, k), dtype=torch.int32, device=device),
                   torch.empty((T, k), dtype=torch.float32, device=device),
                   torch.empty(1, dtype=torch.float32, device=device),
                   torch.empty((T, k), dtype=torch.uint8, device=device),
                   torch.empty(N, dtype=torch.int32, device=device),
                   torch.empty(N, dtype=torch.int32, device=device))


def route(cfg: MoECfg, x: torch.Tensor, w_router: torch.Tensor,
          router_bias: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
          stream=None, options: Optional[Options] = None) -> Routing:
    """moe_route (moe_route_ex with `options`): top-k indices and weights, aux loss,
    capacity drop mask, counts."""
    dt = _io_dtype(cfg)
    _check(x, "x", (cfg.T, cfg.H), dt)
    _check(w_router, "w_router", (cfg.N, cfg.H), dt)
    if router_bias is not None:
        _check(router_bias, "router_bias", (cfg.N,), torch.float32)
    if options is not None:
        options.check(cfg.T)
    if workspace is None:
        workspace = make_workspace(cfg, x.device, options)
    r = _routing_outputs(cfg, x.device)
    args = [_ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(r.topk_idx), _ptr(r.topk_w),
            _ptr(r.aux_loss), _ptr(r.drop_mask), _ptr(r.expert_counts), _ptr(r.kept_counts),
            _ptr(workspace), workspace.numel(), _stream(stream)]
    if options is None:
        rc = library().moe_route(ctypes.byref(cfg), *args)
    else:
        rc = library().moe_route_ex(ctypes.byref(cfg), ctypes.byref(options.to_c()), *args)
    if rc != MOE_OK:
        raise MoEError("moe_route", rc)
    return r


def forward(cfg: MoECfg, x: torch.Tensor, w_router: torch.Tensor,
            router_bias: Optional[torch.Tensor], w1: torch.Tensor, w3: torch.Tensor,
            w2: torch.Tensor, workspace: Optional[torch.Tensor] = None,
            out: Optional[torch.Tensor] = None, routing: Optional[Routing] = None,
            stream=None, stage_events: Optional[Sequence[torch.cuda.Event]] = None,
            options: Optional[Options] = None) -> torch.Tensor:
    """moe_forward (moe_forward_ex with `options`): the layer's MoE branch out[T,H]
    (the caller adds the residual). Pass `routing` (see ``Routing``) to also receive
    the routing outputs. With shared experts w1, w3, w2 hold N + n_shared experts;
    with the GELU expert w3 may be None."""
    dt = _io_dtype(cfg)
    T, H, N, F = cfg.T, cfg.H, cfg.N, cfg.F
    NS = N + (options.n_shared if options is not None else 0)
    gelu = options is not None and options.activation == "gelu"
    _check(x, "x", (T, H), dt)
    _check(w_router, "w_router", (N, H), dt)
    _check(w1, "w1", (NS, F, H), dt)
    if not (gelu and w3 is None):
        _check(w3, "w3", (NS, F, H), dt)
    _check(w2, "w2", (NS, H, F), dt)
    if router_bias is not None:
        _check(router_bias, "router_bias", (N,), torch.float32)
    if options is not None:
        options.check(T)
    if workspace is None:
        workspace = make_workspace(cfg, x.device, options)
    if out is None:
        out = torch.empty((T, H), dtype=dt, device=x.device)
    else:
        _check(out, "out", (T, H), dt)
    r = routing
    args = [_ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(out),
            _ptr(r.topk_idx) if r else None, _ptr(r.topk_w) if r else None,
            _ptr(r.aux_loss) if r else None, _ptr(r.drop_mask) if r else None,
            _ptr(r.expert_counts) if r else None, _ptr(r.kept_counts) if r else None,
            _ptr(workspace), workspace.numel(), _stream(stream)]
    handles = None
    if stage_events is not None:
        if len(stage_events) != MOE_NUM_STAGES + 1:
            raise ValueError(f"stage_events needs {MOE_NUM_STAGES + 1} events")
        handles = (ctypes.c_void_p * len(stage_events))(*[e.cuda_event for e in stage_events])
    if options is not None:
        rc = library().moe_forward_ex(ctypes.byref(cfg), ctypes.byref(options.to_c()), *args,
                                      handles)
    elif handles is None:
        rc = library().moe_forward(ctypes.byref(cfg), *args)
    else:
        rc = library().moe_forward_timed(ctypes.byref(cfg), *args, handles)
    if rc != MOE_OK:
        raise MoEError("moe_forward", rc)
    return out


def new_routing(cfg: MoECfg, device=None) -> Routing:
    return _routing_outputs(cfg, device or "cuda")


def get_status(workspace: torch.Tensor, stream=None) -> int:
    """moe_get_status: synchronise, read and clear the status word; raises when a
    kernel reported a failure."""
    bits = ctypes.c_uint32(0)
    rc = library().moe_get_status(_ptr(workspace), workspace.numel(), _stream(stream),
                                  ctypes.byref(bits))
    if rc != MOE_OK:
        raise MoEError(f"moe_get_status (bits {bits.value:#x})", rc)
    return bits.value


def make_stage_events(stream=None) -> list:
    """MOE_NUM_STAGES+1 timing events, each recorded once so the handle exists."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(MOE_NUM_STAGES + 1)]
    s = stream or torch.cuda.current_stream()
    for e in evs:
        e.record(s)
    return evs


@dataclass
class DeviceInputs:
    x: torch.Tensor
    w_router: torch.Tensor
    router_bias: Optional[torch.Tensor]
    w1: torch.Tensor
    w3: torch.Tensor
    w2: torch.Tensor


def to_torch(a, dtype: str) -> torch.Tensor:
    """A host storage array (bf16 bits as uint16, or float32) as a CPU torch tensor."""
    import numpy as np
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))


def router_weight_to_device(w_router_hn, dtype: str, device="cuda") -> torch.Tensor:
    """A router weight given as W_r [H, N] (logits = x @ W_r) in the library's
    nn.Linear layout [N, H]."""
    import numpy as np
    return to_torch(np.ascontiguousarray(np.asarray(w_router_hn).T), dtype).to(device)


def to_device(inp, device="cuda") -> DeviceInputs:
    """Copy an inputs.MoEInputs to the GPU in the library's layouts (the router weight,
    drawn as W_r [H, N], goes over as [N, H])."""
    def up(a):
        return None if a is None else to_torch(a, inp.dtype).to(device)
    bias = None if inp.router_bias is None else torch.from_numpy(inp.router_bias).to(device)
    return DeviceInputs(up(inp.x), router_weight_to_device(inp.w_router, inp.dtype, device),
                        bias, up(inp.w1), up(inp.w3), up(inp.w2))
