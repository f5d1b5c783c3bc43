"""GB300-native (sm_103a) IO-aware exact attention.

The compute path is ``libfa.so`` (hand-written CUDA for sm_103a behind a C
ABI, declared in ``include/fa.h``); ``exact_io_aware_05_gb300.fa`` is the thin
ctypes binding over it.  Importing this package does not load the library;
importing ``.fa`` does, and fails loudly if it has not been built.
"""
__version__ = "0.1.0"
