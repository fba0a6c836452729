"""CPU oracle of the ZeRO-3 sharded mixed-precision AdamW step.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
baseline leg of the benchmark may import this package.  It shares no code with
the CUDA library and never imports it.
"""
from .zero3_oracle import *  # noqa: F401,F403
