"""CPU oracle of the SPIN indexer step -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and the CPU-baseline leg of bench.py may import
this package.  The CUDA library never does, and this package never imports it.
"""
