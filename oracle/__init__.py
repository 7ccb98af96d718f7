"""CPU oracle for the ONNX matrix-product family (TEST INFRASTRUCTURE ONLY).

This package is the slow, obviously-correct reference that the CUDA library is
checked against.  It is written from the operator pages alone and shares no
code with the CUDA path: nothing under ``quantized_gemm_gb300/`` may import it,
and it imports nothing from there.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

Arithmetic conventions (readings of points the pages leave open):

* Floating point: every input is widened exactly to float64 and the
  contraction is done in float64; results are returned unrounded (float64).
* Integers: contractions are exact modulo 2**64 (uint64 arithmetic) and then
  reduced modulo 2**n of the operator's type T, i.e. numpy's wrap-around.
* QLinearMatMul: the int32 accumulator is the exact integer sum reduced
  modulo 2**32; the requantisation is a fixed sequence of IEEE float32
  operations (see ``qlinear_matmul``).

Each module cites the page and section it follows:

* ``matmul``          -- MatMul (onnx-light, ai.onnx since version 13)
* ``gemm``            -- Gemm (onnx-light, ai.onnx since version 13)
* ``qlinear_matmul``  -- QLinearMatMul - version 10 (onnx-light)
* ``grouped_matmul``  -- GroupedMatMul - 29 (onnx.ai)
* ``dequantize_linear`` -- GroupedMatMul - 29, Summary: weight-only quantized
  experts (DequantizeLinear of the weights, then GroupedMatMul)

A second, independent oracle restates the same pages as plain C++ loops
(``csrc/oracle.cpp``: double accumulation in k order without fused
multiply-adds, exact integers, the same float32 requantisation), bound by
``oracle.native`` with the same function names; it is what the benchmark's CPU
baseline times and what the full-size GPU parity tests use.  The two share no
code.

Parity status: every function of both oracles is pinned by tests in
``tests/test_oracle_pins.py`` (printed worked examples, brute force on tiny
inputs, closed forms, identities and hand-computed error-bound denominators),
and ``tests/test_oracle_native.py`` checks that the two agree on random
inputs; none is "parity unpinned".
"""

from .matmul import matmul, matmul_output_shape, matmul_abs_scale
from .gemm import gemm, gemm_output_shape, gemm_abs_scale
from .qlinear_matmul import qlinear_matmul, requantize
from .grouped_matmul import grouped_matmul, grouped_abs_scale
from .dequantize_linear import (dequantize_linear, unpack_4bit, grouped_matmul_qweights, grouped_qweights_abs_scale,
                                round_to, round_to_bf16)

__all__ = [
    "matmul", "matmul_output_shape", "matmul_abs_scale",
    "gemm", "gemm_output_shape", "gemm_abs_scale",
    "qlinear_matmul", "requantize",
    "grouped_matmul", "grouped_abs_scale",
    "dequantize_linear", "unpack_4bit", "grouped_matmul_qweights", "grouped_qweights_abs_scale", "round_to", "round_to_bf16",
]
