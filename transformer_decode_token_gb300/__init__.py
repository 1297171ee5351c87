"""GPT-2 single-token decode on one GB300 (sm_103a).

The compute path is the CUDA library ``libgpt2.so`` built from ``csrc/``;
``binding`` is a thin ctypes layer over its C ABI (include/gpt2.h).
``synth`` makes the seeded synthetic weights and prompts.  Nothing here is
imported eagerly, so importing ``synth`` alone never loads the CUDA library.
"""
__all__ = ["binding", "synth"]
