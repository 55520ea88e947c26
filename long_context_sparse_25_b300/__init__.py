"""CSA / HCA forward pass for B300 (sm_103a): a C-ABI CUDA library
(``libcsa_b300.so``, header ``include/csa.h``) with a thin ctypes binding
(``long_context_sparse_25_b300.csa``), seeded synthetic inputs
(``.synth``) and a step runner (``.pipeline``)."""
