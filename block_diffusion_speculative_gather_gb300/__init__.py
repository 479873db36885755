"""DFlash block-diffusion speculative-decoding round for GB300 (sm_103a).

Submodules: ``configs`` (the workloads), ``synth`` (seeded synthetic inputs),
``capi`` (ctypes binding of libdflash.so, loaded on import) and ``runtime``
(the PyTorch-side harness).  ``capi``/``runtime`` need the built library.
"""
