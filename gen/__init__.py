"""Seeded synthetic input generators for the tests and the benchmark.

Not part of the library: the shipped package (speculative_decoding_tree_build_gb300)
never imports this. Both the CUDA path and the CPU oracle are fed from here.
"""
