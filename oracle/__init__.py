"""Test infrastructure: the fp64 CPU oracle of one Kimi-K2 MLA layer.  Only tests, the smoke
check and the benchmark's CPU-baseline leg may import this package."""
