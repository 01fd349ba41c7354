"""GB300-native batch-invariant shared LoRA delta operator.

The operator runs in hand-written sm_103a CUDA kernels behind a C ABI
(``include/lora_delta.h``); ``lora_delta`` is its thin ctypes binding.
"""
