"""GB300-native LoRA adapter product: the C ABI liblora.so (include/lora.h) with
hand-written sm_103a kernels, and its thin Python binding.

    from lora_rank_adapter_gb300 import binding as lora
    lora.lora_forward(X, A, B, Y, scale)           # Y += scale * (X @ A) @ B

`synth` draws the seeded synthetic workloads.  `_build.build()` compiles the
library in-tree.
"""
from . import binding, synth  # noqa: F401
from .binding import (LoraError, lora_apply_linear, lora_backward_db, lora_backward_dx_da,  # noqa: F401
                      lora_device_error, lora_expand, lora_forward, lora_gather_shrink,
                      lora_group_by_slot, lora_shrink, lora_version)
