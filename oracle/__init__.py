"""fp64 CPU oracle for paged-KV decode attention, kv append and block copy.

TEST INFRASTRUCTURE ONLY: tests/, the smoke check and the benchmark's CPU
baseline leg import it; the product package never does.
"""
