"""GroupedMatMul oracle (test infrastructure only).

Follows "GroupedMatMul - 29" (onnx.ai operator page): the Summary, Inputs,
Outputs and Type Constraints sections.

* input [M, K], weights [G, K, N], group_indices [M, S], optional bias [G, N];
  output [M, S, N].
* output[m, i] = input[m] @ weights[group_indices[m, i]], plus
  bias[group_indices[m, i]] when bias is present.
* Every index must lie in [0, G); anything else (negative values included) is
  invalid input with undefined behaviour, and negative values do not count
  back from G.  The oracle raises IndexError on such input.
* T is bfloat16, float16, float or double; Tind is int32 or int64.

The page defines the result through a Gather / Expand / MatMul decomposition;
the direct loop over (m, i) below is the same mathematics written per output
row.  Float inputs are widened exactly to float64 and the result is float64,
unrounded; the bias is added to the float64 row sum.
"""

import numpy as np

from ._numeric import to_f64


def _check(input, weights, group_indices, bias):
    if input.ndim != 2 or weights.ndim != 3 or group_indices.ndim != 2:
        raise ValueError("expected input [M,K], weights [G,K,N], group_indices [M,S]")
    M, K = input.shape
    G, K2, N = weights.shape
    if K2 != K or group_indices.shape[0] != M:
        raise ValueError("shape mismatch")
    if group_indices.dtype not in (np.dtype(np.int32), np.dtype(np.int64)):
        raise TypeError("group_indices must be int32 or int64")
    if bias is not None and bias.shape != (G, N):
        raise ValueError("bias must have shape [G, N]")
    return M, K, G, N, group_indices.shape[1]


def grouped_matmul(input, weights, group_indices, bias=None):
    """output[m, i, :] = input[m, :] @ weights[g, :, :] (+ bias[g, :]),  g = group_indices[m, i]."""
    input = np.asarray(input)
    weights = np.asarray(weights)
    group_indices = np.asarray(group_indices)
    bias = None if bias is None else np.asarray(bias)
    M, K, G, N, S = _check(input, weights, group_indices, bias)
    out = np.zeros((M, S, N), dtype=np.float64)
    x = to_f64(input)
    for m in range(M):
        for i in range(S):
            g = int(group_indices[m, i])
            if not 0 <= g < G:
                raise IndexError("group index %d at (%d, %d) is outside [0, %d)" % (g, m, i, G))
            row = x[m] @ to_f64(weights[g])
            if bias is not None:
                row = row + to_f64(bias[g])
            out[m, i] = row
    return out


def grouped_abs_scale(input, weights, group_indices, bias=None):
    """|input[m]| @ |weights[g]| + |bias[g]| in float64: the float error-bound denominator."""
    input = np.abs(to_f64(np.asarray(input)))
    weights = np.abs(to_f64(np.asarray(weights)))
    b = None if bias is None else np.abs(to_f64(np.asarray(bias)))
    return grouped_matmul(input, weights, np.asarray(group_indices), b)
