"""GB300-native batched LLM sampling and speculative verification.

The compute path is a C-ABI shared library of sm_103a CUDA kernels
(``csrc/``, declared in ``include/ss.h``); ``speculative_verification_gb300.ss``
is its thin ctypes binding.  ``workloads`` builds seeded synthetic inputs.
"""
