"""Gemma-4 26B-A4B sparse MoE feed-forward block on one GB300 (sm_103a).

The block runs in hand-written CUDA kernels behind the C ABI declared in include/moe_ffn.h.
``binding`` is the thin ctypes layer over that library (argument marshalling only); ``synth``
draws seeded synthetic inputs. Importing the package loads nothing; the CUDA library is loaded on
first use and its absence is an error, never a fallback.
"""
__all__ = ["binding", "synth"]
