"""CPU oracle for the routed ReLU^2 MoE layer.

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and
by the CPU-baseline leg of bench.py, never by the product path.  It shares no
code with the CUDA library (routed_relu_expert_gb300/) and neither imports the
other.
"""
from . import moe_oracle  # noqa: F401
