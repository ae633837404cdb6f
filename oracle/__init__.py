"""Plain CPU oracle for the block-scaled low-precision matrix multiply.

This package is TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it.  The CUDA library never calls it, and it imports nothing from the CUDA
library or its Python binding: the two share no code.

It restates, in slow and obviously checkable NumPy, what the four source pages
define:

* ``formats``  -- every element and scale format (E4M3, E5M2, E2M1, UE8M0,
  UE4M3) built by enumerating its codes from the sign/exponent/mantissa
  definition, plus nearest-even encoding with saturation.
* ``quantize`` -- the absmax block quantizer: per-block scale from the block's
  largest magnitude, then the codes (atrex-bench #002 block_scaled_mm, Input
  Generation; TensorTonic "Int8 Matmul with Per-Channel Scales", problem
  statement; the UE8M0 / UE4M3 rules are readings, see the function docs).
* ``gemm``     -- the matmul definitions: jax.nn.scaled_matmul's repeat-then-
  einsum definition, block_scaled_mm's per-K-block formulation, the INT8
  per-channel matmul with an exact integer sum, and the MXFP8 linear backward
  of the NKI "Matmul MXFP8 Backward Kernel API Reference".

Floating point: quantizer arithmetic is binary32, as on the pages (their inputs,
scales and quotients are float32 tensors); matmul arithmetic is float64.

Parity status of each function is stated in its docstring.  Two rules have no
value printed on the pages to pin them to (UE8M0 and UE4M3 scale selection);
they are pinned to their defining inequalities and to torch's own E8M0 / E4M3
conversions instead, which the tests check.
"""

from . import formats, quantize, gemm  # noqa: F401
