"""GB300-native multi-LoRA mixed-batch adapter update (SGMV / BGMV / fused layer).

The compute path is a C-ABI CUDA library (``csrc/``, declared in
``include/lora.h``); ``segmented_gathered_rank_gb300.lora`` is its thin
ctypes binding.  Importing this package does not load the library; importing
``lora`` does, and fails loudly when it has not been built.
"""
__all__ = ["inputs", "lora"]
