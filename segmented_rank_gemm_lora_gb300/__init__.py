"""Multi-adapter segmented-rank LoRA for GB300 (sm_103a).

The compute lives in the CUDA library ``liblora.so`` behind the C ABI declared
in ``include/lora.h``; ``segmented_rank_gemm_lora_gb300.lora`` is the thin
ctypes binding over it.  ``synth`` draws seeded synthetic inputs.
"""
