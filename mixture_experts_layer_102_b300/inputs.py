"""Seeded synthetic inputs for the MoE FFN layer, shared by the CUDA path's tests,
the benchmark and the oracle's tests.

The recipe (one numpy PCG64 stream per tensor, spawned from ``SeedSequence(seed)`` in
the order x, router weight, router bias, W1, W3, W2):

* x[T,H] ~ N(0, 1)
* router weight W_r[H,N] ~ N(0, 0.02**2)          (std 0.02)
* W1[N,F,H], W3[N,F,H] ~ N(0, 1/H)                 (std = fan_in**-0.5, fan_in = H)
* W2[N,H,F] ~ N(0, 1/F)                            (std = fan_in**-0.5, fan_in = F)
* optional router bias b[N] = 2.0 * r**-1.1 with r a seeded permutation of 1..N, so
  the hottest expert gets exactly +2.0 (a Zipf(1.1) profile scaled to 2.0 max).
* with ``n_shared`` shared experts the expert tensors hold N + n_shared experts drawn
  from the same streams (the first N are the routed experts' weights unchanged).
* inputs with separated router logits (``make_separated_inputs``), for checking
  routing decisions exactly: W_r is the identity on the first N hidden dims and zero
  elsewhere, x[t, :N] is a seeded permutation of 0, 1/64, ..., (N-1)/64 (exact in
  bf16), the rest of x as above, and the optional bias is the Zipf profile rounded
  to multiples of 1/128. Every logit is then an exact multiple of 1/128, so two
  different logits differ by at least 1/128 and equal ones are equal on every side.
* a valid-token mask (``make_valid_mask``): the batch is cut into sequences of
  ``seq_len`` tokens; sequence b keeps its first L_b tokens, L_b uniform on
  [0, seq_len], and the rest is padding.

Values are drawn as float32 normals. For bf16 workloads every tensor except the
bias is rounded to bf16 (round to nearest even) and the rounded values are what both
the GPU path and the oracle consume. Expert weights use the ``nn.Linear`` [out, in]
orientation, so W1/W3 rows are indexed by the SwiGLU column f and W2 rows by the
hidden column h.

This module draws numbers and converts storage formats; it holds none of the layer's
arithmetic.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import Optional

import numpy as np

from .configs import MoEConfig


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); return the bits.
    Large arrays are converted in chunks on a few threads (same result)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    flat = u.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)

    def part(lo, hi):
        v = flat[lo:hi]
        lsb = (v >> np.uint32(16)) & np.uint32(1)
        out[lo:hi] = (v + np.uint32(0x7FFF) + lsb) >> np.uint32(16)

    chunk = 1 << 24
    if flat.size <= chunk:
        part(0, flat.size)
    else:
        with ThreadPoolExecutor(max_workers=8) as ex:
            list(ex.map(lambda lo: part(lo, min(lo + chunk, flat.size)),
                        range(0, flat.size, chunk)))
    return out.reshape(u.shape)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to the float32 values they encode (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


@dataclass
class MoEInputs:
    """Storage arrays of one layer instance.

    For ``dtype == "bf16"`` the arrays x, w_router, w1, w3, w2 hold uint16 bf16 bit
    patterns; for ``"f32"`` they hold float32. ``router_bias`` is float32 or None.
    """
    dtype: str
    x: np.ndarray
    w_router: np.ndarray
    router_bias: Optional[np.ndarray]
    w1: np.ndarray
    w3: np.ndarray
    w2: np.ndarray

    def values(self, name: str) -> np.ndarray:
        """float32 values of a storage array (bf16 bits widened exactly)."""
        a = getattr(self, name)
        if a is None:
            return None
        if self.dtype == "bf16" and a.dtype == np.uint16:
            return bf16_bits_to_f32(a)
        return a


def _normal(seq: np.random.SeedSequence, shape, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seq))
    out = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def _store(a: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(a) if dtype == "bf16" else a


def make_x(cfg: MoEConfig, rank: int = 0) -> np.ndarray:
    """Activations only. Rank 0 uses the workload's own x stream; rank r > 0 of a
    data-parallel run draws an independent batch from ``SeedSequence([seed, 1000+r])``."""
    seqs = np.random.SeedSequence(cfg.seed).spawn(6)
    seq = seqs[0] if rank == 0 else np.random.SeedSequence([cfg.seed, 1000 + rank])
    return _store(_normal(seq, (cfg.T, cfg.H), 1.0), cfg.dtype)


def make_valid_mask(T: int, seq_len: int, seed: int) -> np.ndarray:
    """[T] uint8, 1 for real tokens: padded sequences of ``seq_len`` tokens."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 2000])))
    n_seq = -(-T // seq_len) if T else 0
    lengths = g.integers(0, seq_len + 1, size=n_seq)
    pos = np.arange(T) % seq_len
    return (pos < lengths[np.arange(T) // seq_len]).astype(np.uint8) if T else \
        np.zeros(0, np.uint8)


def make_inputs(cfg: MoEConfig, rank: int = 0, with_experts: bool = True,
                n_shared: int = 0) -> MoEInputs:
    seqs = np.random.SeedSequence(cfg.seed).spawn(6)
    T, H, N, F = cfg.T, cfg.H, cfg.N, cfg.F
    NE = N + n_shared
    x = make_x(cfg, rank)
    w_router = _store(_normal(seqs[1], (H, N), 0.02), cfg.dtype)
    bias = None
    if cfg.zipf_bias:
        g = np.random.Generator(np.random.PCG64(seqs[2]))
        r = g.permutation(N).astype(np.float64) + 1.0
        bias = (2.0 * r ** -1.1).astype(np.float32)
    if with_experts:
        # one stream per tensor, so the three draws may run side by side
        jobs = [(seqs[3], (NE, F, H), H ** -0.5), (seqs[4], (NE, F, H), H ** -0.5),
                (seqs[5], (NE, H, F), F ** -0.5)]
        with ThreadPoolExecutor(max_workers=3) as ex:
            w1, w3, w2 = ex.map(lambda j: _store(_normal(*j), cfg.dtype), jobs)
    else:
        w1 = w3 = w2 = None
    return MoEInputs(cfg.dtype, x, w_router, bias, w1, w3, w2)


def make_separated_inputs(cfg: MoEConfig, n_shared: int = 0) -> MoEInputs:
    """Inputs whose router logits are exact multiples of 1/128 (see the header)."""
    if cfg.N > cfg.H or cfg.N > 128:
        raise ValueError("separated logits need N <= H and N <= 128")
    base = make_inputs(cfg, n_shared=n_shared)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg.seed, 3000])))
    T, H, N = cfg.T, cfg.H, cfg.N
    x = base.values("x").copy()
    if T:
        x[:, :N] = np.argsort(g.random((T, N)), axis=1).astype(np.float32) / np.float32(64.0)
    w_router = np.zeros((H, N), dtype=np.float32)
    w_router[:N, :N] = np.eye(N, dtype=np.float32)
    bias = None
    if base.router_bias is not None:
        bias = (np.round(base.router_bias.astype(np.float64) * 128.0) / 128.0).astype(np.float32)
    return MoEInputs(cfg.dtype, _store(x, cfg.dtype), _store(w_router, cfg.dtype), bias,
                     base.w1, base.w3, base.w2)
