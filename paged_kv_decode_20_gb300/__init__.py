"""GB300-native paged-KV decode attention (XQA-style call and MLA latent variant).

The compute lives in a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/xqa.h``); ``xqa`` is its thin ctypes
binding.  ``workloads`` draws seeded synthetic inputs.
"""
