"""NVFP4 weight-only SwiGLU FFN decode for GB300 (sm_103a).

The compute lives in the C-ABI library libnvfp4ffn.so (hand-written CUDA);
`nvfp4_weight_only_gb300.ffi` is the thin ctypes binding over it.  Importing
this package loads nothing; the binding loads the library on first use and
raises if it is missing.
"""
