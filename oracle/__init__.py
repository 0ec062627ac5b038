"""fp64 CPU oracle of the top-k routed MoE FFN forward pass.

Test infrastructure only: imported by the tests, the smoke check and the benchmark's
CPU-baseline leg, never by the CUDA product path.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import OracleResult, moe_forward, route  # noqa: F401
