"""CPU oracle for the W4A16 group-quantized linear layer.

TEST INFRASTRUCTURE ONLY. The oracle exists to check the CUDA path; it is not
part of it. Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` leg of ``bench.py`` may import, call or
run anything in this package. The library (``weight_only_bit_04_b300``) never
imports it, and this package imports nothing from the library.

Two independent implementations live here:

* ``w4a16_oracle`` -- NumPy, fp64 throughout: round-to-nearest group
  quantization, canonical 4-bit packing, dequantization and the
  dequantize-then-matmul reference with its per-element error bound.
* ``brute`` -- pure-Python scalar loops (``struct``'s half-precision packing
  for fp16 rounding, Python floats for fp64) for tiny shapes, used to pin
  ``w4a16_oracle`` to something other than itself.

Sources (web pages on 4-bit weight-only quantization):

* "AWQ + GPTQ Quantization, in depth" -- section "What W4A16 buys and why
  decoding gets faster" (4-bit weights, 16-bit activations, one fp16 scale and
  a 4-bit zero point per group of 128 neighbouring input columns) and "The two
  algorithms, compactly" (W is out x in; act order quantizes columns by
  descending diag(H)).
* "LLM Quantization: A Deep Dive into GPTQ, AWQ, and Post-Training
  Quantization" -- section "The Math of Quantization" (q = round(x/S) + Z and
  x ~ (q - Z) * S).
* "LLM Quantization: INT8, GPTQ, and AWQ Explained" -- section "What
  quantization actually does" (find the range, pick the scale, round to the
  nearest grid point; torch.round then clamp; per-group scales).
"""

from . import w4a16_oracle  # noqa: F401
from . import brute  # noqa: F401
