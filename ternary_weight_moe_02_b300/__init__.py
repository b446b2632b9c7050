"""Ternary mixture-of-experts FFN step for B300 (sm_103a).

The CUDA library ``libmaple.so`` (C-ABI declared in ``include/maple.h``) does all of
the work; ``ternary_weight_moe_02_b300.maple`` is its thin ctypes binding.  Importing
the binding fails loudly when the library has not been built.
"""
__all__ = ["maple", "synth"]
