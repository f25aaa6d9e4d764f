"""fp64 CPU oracle for Nyström self-attention (test infrastructure only).

Only the tests, the package's smoke() check and the benchmark's CPU-baseline
leg may import this package. The CUDA library shares no code with it.
"""
