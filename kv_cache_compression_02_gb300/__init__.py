"""CacheGen KV-cache codec for GB300 (sm_103a).

The codec is a C-ABI CUDA library (``libcachegen.so``: ``cg_fit_tables``,
``cg_encode``, ``cg_decode``); :mod:`.cachegen` is its thin ctypes binding.
Importing the package itself loads nothing; the binding loads the library on
first use and raises if it has not been built.
"""
__all__ = ["cachegen", "synth", "workloads"]
