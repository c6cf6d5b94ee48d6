"""GB300-native per-unit FSDP cycle: shard layout, gather+cast, reduce-scatter, AdamW.

The compute path is the C-ABI CUDA library built from ``csrc/`` (see
``include/fsdp_unit.h``); ``binding`` marshals arguments to it.  There is no
CPU fallback: calling into the library without the built extension raises.
"""
