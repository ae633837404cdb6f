"""Pins of the oracle's matmuls: the jax.nn.scaled_matmul basic case (golden),
integer-sum identities, chunked = unchunked, brute-force loops, one-hot scale
index checks, transposition identities and the exact MXFP8 backward on
losslessly representable inputs."""

import json
import os

import numpy as np
import pytest

from oracle import formats as F
from oracle import gemm as G
from oracle import quantize as Q
from tests.conftest import GOLDEN


def test_jax_basic_case():
    with open(os.path.join(GOLDEN, "jax_scaled_matmul_basic.json")) as f:
        ex = json.load(f)
    y = G.scaled_matmul(ex["a"], ex["b"], ex["a_scales"], ex["b_scales"])
    np.testing.assert_array_equal(y, ex["y"])


def test_block_size_inference_and_rejection():
    assert G.block_size(64, 4) == 16             # the cuDNN example's shapes
    assert G.block_size(8192, 256) == 32
    with pytest.raises(ValueError):
        G.block_size(100, 3)


def test_integer_identity_mxfp8_codes():
    """Integer-valued E4M3 codes with power-of-two scales give exact results."""
    rng = np.random.default_rng(1)
    B, M, N, K = 2, 9, 7, 64
    a = rng.integers(-16, 17, (B, M, K)).astype(np.float32)
    b = rng.integers(-16, 17, (B, N, K)).astype(np.float32)
    ca, cb = F.encode(a, "e4m3"), F.encode(b, "e4m3")
    assert (F.decode(ca, "e4m3") == a).all()     # |v| <= 16 integers are exact
    ea = rng.integers(-3, 4, (B, M, K // 32))
    eb = rng.integers(-3, 4, (B, N, K // 32))
    y = G.scaled_matmul(F.decode(ca, "e4m3"), F.decode(cb, "e4m3"), 2.0 ** ea, 2.0 ** eb)
    a_int = a.astype(np.int64) * (2 ** (ea + 3)).repeat(32, -1)
    b_int = b.astype(np.int64) * (2 ** (eb + 3)).repeat(32, -1)
    exact = np.einsum("bmk,bnk->bmn", a_int, b_int) / 64.0
    np.testing.assert_array_equal(y, exact)


def _bf_scaled_matmul(a, b, sa, sb):
    B, M, K = a.shape
    N = b.shape[1]
    bsa, bsb = K // sa.shape[-1], K // sb.shape[-1]
    y = np.zeros((B, M, N))
    for i in range(B):
        for m in range(M):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    acc += (a[i, m, k] * sa[i, m, k // bsa]) * (b[i, n, k] * sb[i, n, k // bsb])
                y[i, m, n] = acc
    return y


def test_scaled_matmul_brute_force():
    rng = np.random.default_rng(2)
    a = rng.standard_normal((2, 3, 12))
    b = rng.standard_normal((2, 4, 12))
    sa = rng.uniform(0.5, 2, (2, 3, 3))          # block 4
    sb = rng.uniform(0.5, 2, (2, 4, 2))          # block 6: blocks need not agree
    np.testing.assert_allclose(G.scaled_matmul(a, b, sa, sb), _bf_scaled_matmul(a, b, sa, sb),
                               rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("m,n,k,gn,gk", [(5, 256, 384, 128, 128), (3, 64, 64, 16, 32)])
def test_chunked_equals_unchunked(m, n, k, gn, gk):
    rng = np.random.default_rng(m)
    a = rng.standard_normal((m, k))
    b = rng.standard_normal((n, k))
    sa = rng.uniform(0.1, 3, (m, k // gk))
    sb = rng.uniform(0.1, 3, (n // gn, k // gk))
    y = G.grouped_matmul(a, b, sa, sb, gn, gk)
    a_s, b_s = G.grouped_operands(a, b, sa, sb, gn, gk)
    np.testing.assert_allclose(y, a_s @ b_s.T, rtol=1e-12, atol=1e-12)
    # the jax form with the weight scales expanded over n
    y_jax = G.scaled_matmul(a[None], b[None], sa[None], np.repeat(sb, gn, 0)[None])[0]
    np.testing.assert_allclose(y, y_jax, rtol=1e-12, atol=1e-12)


def test_grouped_one_hot_scales():
    """Only the (row, K block) / (n group, K block) with a nonzero scale may
    contribute: pins the floor(k / group_k) and floor(n / group_n) indexing."""
    rng = np.random.default_rng(4)
    m, n, k, gn, gk = 4, 6, 12, 3, 4
    a = rng.standard_normal((m, k))
    b = rng.standard_normal((n, k))
    sa = np.zeros((m, k // gk)); sa[2, 1] = 2.0
    sb = np.zeros((n // gn, k // gk)); sb[1, 1] = 0.5
    y = G.grouped_matmul(a, b, sa, sb, gn, gk)
    expect = np.zeros((m, n))
    expect[2, 3:6] = 2.0 * 0.5 * (a[2, 4:8] @ b[3:6, 4:8].T)
    np.testing.assert_allclose(y, expect, rtol=1e-14, atol=1e-14)


def test_scaled_matmul_one_hot_scales_and_transpose():
    rng = np.random.default_rng(6)
    a = rng.standard_normal((1, 3, 8))
    b = rng.standard_normal((1, 5, 8))
    sa = np.zeros((1, 3, 2)); sa[0, 1, 1] = 1.0
    sb = np.ones((1, 5, 4))
    y = G.scaled_matmul(a, b, sa, sb)
    expect = np.zeros((3, 5)); expect[1] = a[0, 1, 4:] @ b[0, :, 4:].T
    np.testing.assert_allclose(y[0], expect, rtol=1e-14, atol=1e-14)
    sa2 = rng.uniform(0.5, 2, (1, 3, 2))
    np.testing.assert_allclose(G.scaled_matmul(b, a, sb, sa2)[0], G.scaled_matmul(a, b, sa2, sb)[0].T,
                               rtol=1e-14)


def test_entries_match_full():
    rng = np.random.default_rng(8)
    a = rng.standard_normal((2, 7, 64)); b = rng.standard_normal((2, 5, 64))
    sa = rng.uniform(0.5, 2, (2, 7, 2)); sb = rng.uniform(0.5, 2, (2, 5, 4))
    y = G.scaled_matmul(a, b, sa, sb)
    bd = G.scaled_matmul_bound(a, b, sa, sb)
    ib, im, inn = rng.integers(0, 2, 20), rng.integers(0, 7, 20), rng.integers(0, 5, 20)
    e, eb = G.scaled_matmul_entries(a, b, sa, sb, ib, im, inn)
    np.testing.assert_allclose(e, y[ib, im, inn], rtol=1e-13)
    np.testing.assert_allclose(eb, bd[ib, im, inn], rtol=1e-13)
    a2, b2 = a[0], b[0]
    sa2 = rng.uniform(0.5, 2, (7, 2)); sb2 = rng.uniform(0.5, 2, (1, 2))
    yg = G.grouped_matmul(a2, b2, sa2, sb2, 5, 32)
    e2, _ = G.grouped_entries(a2, b2, sa2, sb2, 5, 32, im, inn)
    np.testing.assert_allclose(e2, yg[im, inn], rtol=1e-13)


def test_int8_sum_bound_and_zero():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((6, 64)).astype(np.float32)
    w = rng.standard_normal((64, 6)).astype(np.float32)
    x[2] = 0; w[:, 4] = 0
    out = G.int8_channel(x, w)
    assert np.abs(out["acc"]).max() <= 64 * 127 * 127
    assert (out["y"][2] == 0).all() and (out["y"][:, 4] == 0).all()
    assert out["x_scales"][2] == 1 and out["w_scales"][4] == 1
    np.testing.assert_array_equal(out["acc"], out["x_q"].astype(np.int64) @ out["w_q"].astype(np.int64))


def test_backward_exact_on_representable_inputs():
    """Entries in {0, +-1, +-2}: every E5M2 code and UE8M0 scale is exact, so
    dX and dW equal the exact integer products.  M != N != K pins the
    transposes."""
    rng = np.random.default_rng(12)
    M, N, K = 64, 96, 32
    dY = rng.integers(-2, 3, (M, N)).astype(np.float32)
    W = rng.integers(-2, 3, (N, K)).astype(np.float32)
    X = rng.integers(-2, 3, (M, K)).astype(np.float32)
    out = G.linear_backward(dY, W, X)
    np.testing.assert_array_equal(out["dX"], dY.astype(np.float64) @ W)
    np.testing.assert_array_equal(out["dW"], dY.T.astype(np.float64) @ X)
    assert out["dy_n_s"].shape == (M, N // 32) and out["wt_s"].shape == (K, N // 32)
    assert out["dyt_s"].shape == (N, M // 32) and out["xt_s"].shape == (K, M // 32)
    assert out["wt"].shape == (K, N) and out["dyt"].shape == (N, M) and out["xt"].shape == (K, M)


def test_backward_close_to_float_product():
    """Random values: within the E5M2 quantization error of the exact product
    (each operand's relative error is at most 2**-3)."""
    rng = np.random.default_rng(13)
    M, N, K = 64, 64, 96
    dY = rng.standard_normal((M, N)).astype(np.float32)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    X = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    out = G.linear_backward(dY, W, X)
    tol = (2 * 2.0 ** -3 + 2.0 ** -6) * (np.abs(dY) @ np.abs(W))
    assert (np.abs(out["dX"] - dY.astype(np.float64) @ W) <= tol).all()
    tolw = (2 * 2.0 ** -3 + 2.0 ** -6) * (np.abs(dY.T) @ np.abs(X))
    assert (np.abs(out["dW"] - dY.T.astype(np.float64) @ X) <= tolw).all()
    # bound is the sum of magnitudes of the dequantized products
    assert (out["dX_bound"] >= np.abs(out["dX"]) - 1e-9).all()


def test_within_bound_rejects_planted_error():
    y_ref = np.array([1.0, -2.0]); bound = np.array([10.0, 10.0])
    assert G.within_bound(y_ref + 0.019, y_ref, bound).all()
    assert not G.within_bound(y_ref + 0.021, y_ref, bound).all()


def test_bf16_output_rounding_allowance_is_half_an_ulp():
    """Rounding to bfloat16 may move a value by up to 2**-8 of it: 16447.25
    rounds to 16384 (spacing 128 there); the allowance admits exactly that and
    no more."""
    import torch
    v = 16447.25
    r = torch.tensor([v]).to(torch.bfloat16).float().item()
    assert r == 16384.0
    assert G.within_bound(np.array([r]), np.array([v]), np.array([0.0]), out_round=G.BF16_HALF_ULP).all()
    assert not G.within_bound(np.array([r - 1]), np.array([v]), np.array([0.0]), out_round=G.BF16_HALF_ULP).all()


def test_dequantize_matches_scaled_operand():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    c, s = Q.quantize(x, (1, 32), "e4m3", "ue8m0")
    d = Q.dequantize(c, s, (1, 32), "e4m3", "ue8m0")
    np.testing.assert_array_equal(d, G.scaled_operand(F.decode(c, "e4m3"), F.decode(s, "ue8m0")))
