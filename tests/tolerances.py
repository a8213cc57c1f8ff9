"""Parity tolerances of the GPU tests.

TOL: floating-point values within TOL times the row's largest magnitude
(the stated rule: 2e-2 for bf16, 1e-4 for fp32).

bf16 final hidden rows (the output of five bf16 layers) use a rule derived in
tests/test_bf16_tolerance.py from an fp32 implementation of the oracle's own
arithmetic: relative L2 error <= BF16_HIDDEN_L2 and max-abs error <=
BF16_HIDDEN_MAXABS_RATIO * BF16_HIDDEN_L2 of the row's largest magnitude.
"""

TOL = {"f32": 1e-4, "bf16": 2e-2}
BF16_HIDDEN_L2 = 2e-2
BF16_HIDDEN_MAXABS_RATIO = 1.5
