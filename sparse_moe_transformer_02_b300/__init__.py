"""B300-native forward pass of one sparse Mixture-of-Experts FFN layer.

The compute lives in ``libmoe.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/moe.h``); ``binding`` is a ctypes layer with the
same function names, and ``inputs`` makes seeded synthetic inputs.
"""
