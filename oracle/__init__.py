"""Plain CPU oracle for batched speculative-decoding verification.

Test infrastructure only: the test suite, the smoke check and the benchmark's
CPU-baseline leg use it; the CUDA product path never does.
"""
