"""CPU oracle for the block-quantized GEMV and grouped-MoE expert path.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or calls this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference leg of ``bench.py`` use it.  It shares no code with the CUDA path.

It is a plain, slow, obviously correct restatement of what the path computes,
in float64 wherever the method does not fix the precision, written from the
Strata pull-request pages:

* #2356 "pf_wmma: a second Volta prompt-expert kernel for IQ2_S gate/up and
  IQ4_NL down" (Summary; Checks) -- IQ4_NL blocks, FP16 prompt experts.
* #1525 "prefill: dense IQ4_XS / Q8_0 to FP16 with 16-byte stores, swiglu +
  q8_1 and the MoE combine ... fused" (Change) -- SwiGLU + q8_1 of H, FP16
  dequantisation by one round-to-nearest-even, the MoE combine.
* #242 "IQ kernels: decode each weight part once for every column and entry,
  bitwise identical" (What it does) -- multi-column GEMV, grouped gate/up and
  down expert GEMVs.
* #1424 "Pascal GP100: a Q8_0 decode GEMV ... and IQ3_XXS / IQ3_S tables in
  shared memory" (What changed) -- Q8_0 GEMV on q8_1 activations, packed planes,
  CPU double reference with relative error below 1e-5.

Modules:
  formats  -- Q8_0 / IQ4_NL block decoding and the IQ4_NL codebook
  q8_1     -- the q8_1 activation quantiser
  gemv     -- per-block integer dots, the multi-column GEMV, its error bound
  moe      -- top-k routing, SwiGLU, the grouped MoE decode layer
  prefill  -- FP16 roundings, expert sort, the grouped MoE prefill layer

Every function states which passage it follows.  Every function is pinned by
the ``-m "not gpu"`` tests in ``tests/test_oracle_*.py`` against closed forms,
brute force on tiny inputs and hand-derived fixtures under ``tests/golden/``.
"""
from . import formats, q8_1, gemv, moe, prefill  # noqa: F401
