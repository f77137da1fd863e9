"""CPU oracle for the bitwise-reproducible optimizer step.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU-baseline
leg are the only callers.  The product path never imports this package.
"""
