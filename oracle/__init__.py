"""fp64 CPU oracle for the speculative-decoding verify step -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import it.
"""
