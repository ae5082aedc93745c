"""fp64 CPU oracle of the tensor-parallel linear block.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, links or runs
this package: only the tests, the smoke check and the benchmark's CPU-baseline
leg may. It shares no code with the CUDA library (no kernels, headers, tables or
helpers); its inputs are plain numpy arrays.

Every function computes the plain definition of one step in float64, with a
library matmul as its only primitive, and cites the passage it follows. Pins
(checks against values and identities that the pages and mathematics fix) live
in tests/test_oracle_pins.py and tests/test_oracle_gpt_pins.py (the vocabulary-
parallel embedding / cross-entropy and the small GPT of `gpt_oracle`). No function
here is "parity unpinned".
"""
from .tp_oracle import *  # noqa: F401,F403
