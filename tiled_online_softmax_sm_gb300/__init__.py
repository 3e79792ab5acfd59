"""GB300 (sm_103a) tiled online-softmax attention.

The compute lives in ``libfa_gb300.so`` (CUDA kernels behind the C ABI of
``include/fa.h``); ``binding`` marshals arguments to it.  ``inputs`` holds the
seeded synthetic input generators.  Importing the package does not load the
library; the first call through ``binding`` does, and raises if it is missing.
"""
