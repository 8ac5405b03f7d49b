"""EvoAttention for GB300 (sm_103a): the memory-efficient 3D attention over the
pair representation (MegaFold's EvoFlash-3D), forward and backward, as
hand-written CUDA kernels behind a C ABI (``include/evoattn.h``).

``protein_folding_attention_gb300.evoattn`` is the Python binding (argument
marshalling only); ``protein_folding_attention_gb300.synthetic`` draws seeded
inputs.  Importing this package loads nothing; the binding loads the CUDA
library on first use and raises if it has not been built.
"""
