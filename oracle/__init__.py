"""CPU oracle for the sparse top-k MoE layer (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this package; the CUDA product path never does.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (ACT_GELU, ACT_RELU, ACT_SWIGLU, GATE_SIGMOID_RENORM,
                         GATE_SOFTMAX_FULL, GATE_SOFTMAX_TOPK)  # noqa: F401
