"""CPU oracle for the gpt-oss MoE MLP block (test infrastructure only).

Only tests/, the smoke entry point and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never does.
"""
from . import moe_oracle  # noqa: F401
