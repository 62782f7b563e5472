"""CPU oracle for the DeepSeekMoE layer forward (test infrastructure only).

Imported only by the tests, the smoke check and the benchmark's CPU-baseline
leg; the product path never touches it.
"""
