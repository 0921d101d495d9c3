"""gather_lora_gb300: routed multi-LoRA fold (bgmv + MoE grouped fold) for GB300.

The compute lives in ``libgather_lora.so`` (hand-written sm_103a CUDA behind a
C ABI declared in ``include/gather_lora.h``). ``gather_lora_gb300.lib`` is the
thin ctypes binding with the same entry-point names; importing this package
does not load the library, and every compute call raises if it is missing.
"""
__all__ = ["lib", "workloads"]
