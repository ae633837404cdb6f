"""Matmul definitions (oracle; test infrastructure).  Arithmetic is float64.

* :func:`scaled_matmul` -- jax.nn.scaled_matmul, the "Mathematically" passage:
  block sizes are ``K // K_a`` and ``K // K_b``; each operand is multiplied by
  its scales repeated along K; the result is ``einsum('BMK,BNK->BMN')``.
* :func:`grouped_matmul` -- atrex-bench #002 block_scaled_mm, Reference
  Implementation: per K block of ``group_k`` the block dot products of the two
  code matrices, scaled by ``a_scales[m, kb] * b_scales[n // group_n, kb]`` and
  summed over the blocks.
* :func:`int8_channel` -- TensorTonic "Int8 Matmul with Per-Channel Scales":
  per-row codes of x, per-column codes of w, the exact integer sum of code
  products, and ``y = a * s_x[b] * s_w[j]``.
* :func:`linear_backward` -- NKI "Matmul MXFP8 Backward Kernel API Reference",
  introduction and Parameters: with ``Y = X @ W^T`` the gradients are
  ``dX = dY @ W`` (contracting N) and ``dW = dY^T @ X`` (contracting M), each
  operand MXFP8-quantized (default float8_e5m2) along its own contraction axis,
  outputs bfloat16.

Every function also exposes the per-entry magnitude sum
``sum_k |a_s[m,k] * b_s[n,k]|`` that the floating-point parity bound scales.
"""

from __future__ import annotations

import numpy as np

from . import formats as F
from . import quantize as Q


def _as64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def block_size(K: int, n_scales: int) -> int:
    """jax.nn.scaled_matmul, Parameters/Notes: K must be a multiple of the
    number of scales along K; the block size is the quotient."""
    if n_scales <= 0 or K % n_scales:
        raise ValueError(f"K={K} is not a multiple of the scale count {n_scales}")
    return K // n_scales


def scaled_operand(v, scales) -> np.ndarray:
    """``v * repeat(scales, K // K_s, axis=-1)`` in float64."""
    v, scales = _as64(v), _as64(scales)
    bs = block_size(v.shape[-1], scales.shape[-1])
    return v * np.repeat(scales, bs, axis=-1)


def scaled_matmul(a, b, a_scales, b_scales) -> np.ndarray:
    """(B,M,K) x (B,N,K) -> (B,M,N) on decoded values and decoded scales."""
    a_s = scaled_operand(a, a_scales)
    b_s = scaled_operand(b, b_scales)
    return np.einsum("bmk,bnk->bmn", a_s, b_s)


def scaled_matmul_bound(a, b, a_scales, b_scales) -> np.ndarray:
    """Per-entry ``sum_k |a_s * b_s|`` for :func:`scaled_matmul`."""
    a_s = np.abs(scaled_operand(a, a_scales))
    b_s = np.abs(scaled_operand(b, b_scales))
    return np.einsum("bmk,bnk->bmn", a_s, b_s)


def scaled_matmul_entries(a, b, a_scales, b_scales, ib, im, in_):
    """Selected entries ``y[ib[i], im[i], in_[i]]`` of :func:`scaled_matmul`,
    each computed on its own as one K-long dot product, with their bounds."""
    ib, im, in_ = (np.asarray(t, dtype=np.int64) for t in (ib, im, in_))
    a_rows = scaled_operand(_as64(a)[ib, im], _as64(a_scales)[ib, im])
    b_rows = scaled_operand(_as64(b)[ib, in_], _as64(b_scales)[ib, in_])
    prod = a_rows * b_rows
    return prod.sum(axis=-1), np.abs(prod).sum(axis=-1)


def grouped_matmul(a, b, a_scales, b_scales, group_n: int, group_k: int) -> np.ndarray:
    """y[m, n] = sum_kb a_scales[m,kb] * b_scales[n//group_n, kb] *
    sum_{k in block kb} a[m,k] * b[n,k]   (a: [m,k], b: [n,k] decoded values)."""
    a, b = _as64(a), _as64(b)
    sa, sb = _as64(a_scales), _as64(b_scales)
    m, k = a.shape
    n = b.shape[0]
    if k % group_k or n % group_n:
        raise ValueError("k must be a multiple of group_k and n of group_n")
    nkb = k // group_k
    if sa.shape != (m, nkb) or sb.shape != (n // group_n, nkb):
        raise ValueError("scale shapes do not match the groups")
    sb_per_n = np.repeat(sb, group_n, axis=0)            # [n, nkb]
    y = np.zeros((m, n), dtype=np.float64)
    for kb in range(nkb):
        ks = slice(kb * group_k, (kb + 1) * group_k)
        dots = a[:, ks] @ b[:, ks].T                       # block partial
        y += dots * sa[:, kb][:, None] * sb_per_n[:, kb][None, :]
    return y


def grouped_operands(a, b, a_scales, b_scales, group_n: int, group_k: int):
    """The scaled operands ``a_s``, ``b_s`` of :func:`grouped_matmul` written
    in the jax.nn.scaled_matmul form (scales repeated along K and over n)."""
    a_s = scaled_operand(a, a_scales)
    sb_per_n = np.repeat(_as64(b_scales), group_n, axis=0)
    b_s = scaled_operand(b, sb_per_n)
    return a_s, b_s


def grouped_entries(a, b, a_scales, b_scales, group_n, group_k, im, in_):
    """Selected entries of :func:`grouped_matmul` and their bounds, one dot
    product each (used for sampled parity at full size)."""
    im, in_ = np.asarray(im, np.int64), np.asarray(in_, np.int64)
    a_rows = scaled_operand(_as64(a)[im], _as64(a_scales)[im])
    b_rows = scaled_operand(_as64(b)[in_], _as64(b_scales)[in_ // group_n])
    prod = a_rows * b_rows
    return prod.sum(axis=-1), np.abs(prod).sum(axis=-1)


def int8_channel(x, w) -> dict:
    """TensorTonic INT8 per-channel matmul on x [B, D_in], w [D_in, D_out].

    Returns the page's dict (``w_q``, ``w_scales``, ``x_q``, ``x_scales``,
    ``y``) plus ``acc`` (the exact integer sums, int64) and ``y_ref``
    (``acc * s_x * s_w`` in float64 from the binary32 scales, which is what the
    page's checker compares ``y`` with)."""
    x_q, x_s = Q.int8_per_row(x)
    w_q, w_s = Q.int8_per_col(w)
    acc = x_q.astype(np.int64) @ w_q.astype(np.int64)
    y_ref = acc.astype(np.float64) * x_s.astype(np.float64)[:, None] * w_s.astype(np.float64)[None, :]
    y32 = (acc.astype(np.float32) * x_s[:, None]) * w_s[None, :]
    return {"w_q": w_q, "w_scales": w_s, "x_q": x_q, "x_scales": x_s,
            "y": y32.astype(np.float32), "acc": acc, "y_ref": y_ref}


def mx_quantize(v, axis: str, fp8: str):
    """MXFP8 quantization of a 2-D binary32 array in 32-element blocks along
    ``axis`` ('cols': blocks run along the contiguous axis, output as is;
    'rows': blocks run down the columns, output transposed so the blocked axis
    becomes contiguous).  UE8M0 scales."""
    if axis == "cols":
        return Q.quantize(v, (1, 32), fp8, "ue8m0", transpose_out=False)
    if axis == "rows":
        return Q.quantize(v, (32, 1), fp8, "ue8m0", transpose_out=True)
    raise ValueError(axis)


def linear_backward(dY, W, X, fp8: str = "e5m2") -> dict:
    """dX = dY @ W and dW = dY^T @ X with MXFP8 operands.

    dY [M, N], W [N, K], X [M, K] are binary32 arrays holding the bfloat16
    inputs' values.  dX contracts N: its left operand is dY blocked along N,
    its right operand W^T [K, N] (W blocked along N, stored transposed).
    dW contracts M: left operand dY^T [N, M] (dY blocked along M, transposed),
    right operand X^T [K, M] (X blocked along M, transposed).  Returns the
    codes and UE8M0 scales of all four operands and the float64 products with
    their per-entry bounds; the bfloat16 rounding of the outputs is left to
    the comparison."""
    dy_n, dy_n_s = mx_quantize(dY, "cols", fp8)       # [M, N], [M, N/32]
    wt, wt_s = mx_quantize(W, "rows", fp8)            # [K, N], [K, N/32]
    dyt, dyt_s = mx_quantize(dY, "rows", fp8)         # [N, M], [N, M/32]
    xt, xt_s = mx_quantize(X, "rows", fp8)            # [K, M], [K, M/32]
    dec = lambda c: F.decode(c, fp8)[None]            # noqa: E731
    sc = lambda s: F.decode(s, "ue8m0")[None]         # noqa: E731
    dX = scaled_matmul(dec(dy_n), dec(wt), sc(dy_n_s), sc(wt_s))[0]
    dX_b = scaled_matmul_bound(dec(dy_n), dec(wt), sc(dy_n_s), sc(wt_s))[0]
    dW = scaled_matmul(dec(dyt), dec(xt), sc(dyt_s), sc(xt_s))[0]
    dW_b = scaled_matmul_bound(dec(dyt), dec(xt), sc(dyt_s), sc(xt_s))[0]
    return {"dy_n": dy_n, "dy_n_s": dy_n_s, "wt": wt, "wt_s": wt_s,
            "dyt": dyt, "dyt_s": dyt_s, "xt": xt, "xt_s": xt_s,
            "dX": dX, "dX_bound": dX_b, "dW": dW, "dW_bound": dW_b}


# Half a unit in the last place of a bfloat16 value, relative (8 significant bits).
BF16_HALF_ULP = 2.0 ** -8


def within_bound(y, y_ref, bound, rel: float = 2e-3, out_round: float = 0.0) -> np.ndarray:
    """Floating-point gate: ``|y - y_ref| <= rel * sum_k |a_s * b_s|``, plus
    ``out_round * |y_ref|`` for the rounding of the output to a narrower type
    (``BF16_HALF_ULP`` for bfloat16 outputs: the NKI backward returns
    bfloat16, and rounding an FP32 result to bfloat16 alone may move it by half
    a bfloat16 ulp, up to 2**-8 of its magnitude)."""
    y_ref = _as64(y_ref)
    return np.abs(_as64(y) - y_ref) <= rel * _as64(bound) + out_round * np.abs(y_ref)
