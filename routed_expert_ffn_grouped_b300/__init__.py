"""B300-native routed MoE FFN layer (int4 g32 experts x q8 activations).

The compute lives in ``libcolibri.so`` (CUDA for sm_103a, C ABI declared in
``include/colibri.h``). ``routed_expert_ffn_grouped_b300.colibri`` is the thin
Python binding with the same entry-point names; ``synth`` draws seeded
synthetic layers. The binding loads the library on first use and raises if it
is missing: there is no CPU fallback.
"""
from . import synth  # noqa: F401

__all__ = ["synth"]
