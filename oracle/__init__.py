"""CPU oracle of the Qwen3 decoder forward (test infrastructure only).

Only tests/, the smoke check and the benchmark's CPU-baseline leg may use it.
"""
