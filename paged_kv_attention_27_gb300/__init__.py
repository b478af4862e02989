"""Paged-KV attention for GB300 (sm_103a): batch decode with GQA and split-KV,
causal variable-length batch prefill, and merge_states, behind the C ABI of
include/fi.h (libfi.so). ``binding`` is the ctypes layer over that library,
``device`` moves synthetic batches (``synth``) to the GPU, ``build`` compiles
the library with nvcc."""
