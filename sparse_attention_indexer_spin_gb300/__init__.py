"""SPIN (Shadow Predictive Indexer) decode-time indexer step for GB300 (sm_103a).

The compute path is the C-ABI library built from csrc/ (libspin.so); `spin` is its thin
ctypes binding and `synthetic` the seeded input generator.  Import the submodules
directly: importing the package itself loads nothing.
"""
__all__ = ["spin", "synthetic"]
