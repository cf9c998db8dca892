"""GB300 (sm_103a) verification path of speculative decoding with layer-skip
self-drafting: hand-written CUDA kernels behind the C ABI in include/spec.h,
compiled into _lib/libspec.so, and a thin ctypes binding (``spec``).

Importing the package loads nothing; ``spec.load()`` (called by every binding
function) loads the compiled library and fails if it is missing.
"""
