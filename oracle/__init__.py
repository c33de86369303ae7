"""CPU oracle of the codebook-4bit matvec: test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package; the product path never does.
"""
