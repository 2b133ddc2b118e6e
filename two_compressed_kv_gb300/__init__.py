"""GB300 (sm_103a) decode attention over a two-D compressed KV cache.

`two_compressed_kv_gb300.mkv` is the ctypes binding of the C ABI declared in
include/mkv.h (libmkv.so, built by `build_lib.build()`); `workloads` holds the
seeded synthetic input recipes.  Importing the package does not load the
library; importing `two_compressed_kv_gb300.mkv` does, and fails loudly when it
is not built.
"""
__all__ = ["mkv", "workloads", "build_lib"]
