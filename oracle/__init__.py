"""CPU oracle of the fused vocabulary-row losses: test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
"""
