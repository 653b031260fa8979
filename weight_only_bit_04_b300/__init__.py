"""W4A16 group-quantized linear layer for NVIDIA B300 (sm_103a).

``w4a16`` is the Python binding of the C-ABI library ``libw4a16.so`` (built
in-tree by ``python -m weight_only_bit_04_b300.build``); ``synth`` holds the
seeded synthetic inputs. The library is loaded on first use and its absence
is an error, never a fallback.
"""

__all__ = ["w4a16", "synth"]
