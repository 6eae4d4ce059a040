"""fp64 CPU oracle for unified paged attention -- TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check in __graft_entry__ and the benchmark's
CPU-baseline leg may import this package.  The CUDA library never links,
loads or calls anything here, and this package imports nothing from it.
"""
