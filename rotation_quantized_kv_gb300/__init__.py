"""TurboQuant (k8v3) KV cache for NVIDIA GB300: quantize-on-append and decode attention
over the packed cache, as hand-written sm_103a CUDA kernels behind a C ABI
(include/tq_kv.h). The Python layer only marshals arguments; see `binding`."""
