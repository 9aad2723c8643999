"""CPU oracle for the activation-sparse MoE path: TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 numpy restatement of what the method computes, written
from "Skipping dead neurons: a faster Nemotron 3.5 Lightning on Apple silicon"
(sevren.ai blog, "Heimr Sparse Down").  Only the tests, the smoke check and the
CPU-baseline leg of the benchmark may import it; the product path never does.
It shares no code with the CUDA library and does not import it.

Every function is pinned by `-m "not gpu"` tests to something other than
itself (hand-worked values, closed forms, brute force on tiny inputs,
invariants); see tests/test_oracle_pins.py.  One figure on the page is not
reproduced and stays "parity unpinned": the 1.3 MB of shared-expert down bytes
quoted in the section "The whole decode step" (the byte model here is pinned
to the page's 5.6 MB and 8.4 GB figures instead).
"""
from .moe import *  # noqa: F401,F403
from .requant import *  # noqa: F401,F403
