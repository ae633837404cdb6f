"""Pins of the oracle's quantizer: the TensorTonic worked examples (golden),
the atrex-bench input generator re-run with torch's own binary32 arithmetic and
float8 conversion, brute-force pure-Python loops on tiny inputs, and the
defining inequalities of the scale rules."""

import json
import math
import os
import struct

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as G
from oracle import quantize as Q
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# TensorTonic worked examples
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("i", [0, 1, 2])
def test_int8_examples(i):
    ex = _golden("int8_per_channel_examples.json")["examples"][i]
    out = G.int8_channel(np.array(ex["x"], np.float32), np.array(ex["w"], np.float32))
    np.testing.assert_array_equal(out["w_q"], ex["w_q"])
    np.testing.assert_array_equal(out["x_q"], ex["x_q"])
    # printed to 6 decimals
    np.testing.assert_allclose(out["w_scales"], ex["w_scales"], rtol=0, atol=0.5e-6)
    np.testing.assert_allclose(out["x_scales"], ex["x_scales"], rtol=0, atol=0.5e-6)
    np.testing.assert_allclose(out["y"], ex["y"], rtol=0, atol=0.5e-6)
    np.testing.assert_allclose(out["y_ref"], ex["y"], rtol=0, atol=0.5e-6)
    if "acc" in ex:
        np.testing.assert_array_equal(out["acc"], ex["acc"])
    # the page's checker: y within 1e-6 relative of acc*sx*sw, zero sum -> exactly 0
    rel = np.abs(out["y"] - out["y_ref"]) <= 1e-6 * np.abs(out["y_ref"])
    assert rel.all()
    assert (out["y"][out["acc"] == 0] == 0).all()


# ----------------------------------------------------------------------------
# atrex-bench input generator, re-run with torch (independent fp32 arithmetic)
# ----------------------------------------------------------------------------

def _torch_generator_recipe(a_raw, b_raw, gn, gk):
    """The atrex-bench recipe in torch ops, with the magnitude maximum for
    both operands (the page takes it without abs for the weights; this
    oracle reads both as the magnitude maximum)."""
    fp8_max = torch.finfo(torch.float8_e4m3fn).max
    n, k = b_raw.shape
    b_max = b_raw.abs().view(n // gn, gn, k // gk, gk).amax(dim=1).amax(dim=-1)
    b_scales = torch.clamp(b_max / fp8_max, min=1e-10)
    b_q = (b_raw / b_scales.repeat_interleave(gn, 0).repeat_interleave(gk, 1)).clamp(-fp8_max, fp8_max)
    b_q = b_q.to(torch.float8_e4m3fn)
    m = a_raw.shape[0]
    a_max = a_raw.abs().view(m, k // gk, gk).amax(dim=-1)
    a_scales = torch.clamp(a_max / fp8_max, min=1e-10)
    a_q = (a_raw / a_scales.repeat_interleave(gk, dim=1)).clamp(-fp8_max, fp8_max).to(torch.float8_e4m3fn)
    return a_q, a_scales, b_q, b_scales


@pytest.mark.parametrize("m,n,k", [(64, 256, 256), (37, 128, 384)])
def test_fp32_scale_matches_torch_recipe(m, n, k):
    g = torch.Generator().manual_seed(m * n + k)
    a_raw = torch.randn(m, k, generator=g)
    b_raw = torch.randn(n, k, generator=g) * 3
    a_raw[3, :128] = 0                            # an all-zero block
    aq, as_, bq, bs = _torch_generator_recipe(a_raw, b_raw, 128, 128)
    codes_a, s_a = Q.quantize(a_raw.numpy(), (1, 128), "e4m3", "f32")
    codes_b, s_b = Q.quantize(b_raw.numpy(), (128, 128), "e4m3", "f32")
    np.testing.assert_array_equal(codes_a, aq.view(torch.uint8).numpy())
    np.testing.assert_array_equal(codes_b, bq.view(torch.uint8).numpy())
    np.testing.assert_array_equal(s_a, as_.numpy())
    np.testing.assert_array_equal(s_b, bs.numpy())
    assert s_a[3, 0] == np.float32(1e-10)         # clamp of the all-zero block


# ----------------------------------------------------------------------------
# Brute force: pure-Python loops with struct-rounded binary32 arithmetic
# ----------------------------------------------------------------------------

def _r32(v: float) -> float:
    return struct.unpack("f", struct.pack("f", v))[0]


def _bf_scale(absmax, code, scale):
    qmax = {"e4m3": 448.0, "e5m2": 57344.0, "e2m1": 6.0, "int8": 127.0}[code]
    r = _r32(absmax / qmax)
    if scale == "f32":
        if code == "int8":
            return 1.0 if absmax == 0 else r
        return max(r, _r32(1e-10))
    if scale == "ue8m0":
        if absmax == 0:
            return 1.0
        # smallest power of two >= r among the 255 UE8M0 values
        cands = [2.0 ** (e - 127) for e in range(255) if 2.0 ** (e - 127) >= r]
        return cands[0] if cands else 2.0 ** 127
    if scale == "ue4m3":
        if absmax == 0:
            return 1.0
        vals = [v for v in F.table("ue4m3") if math.isfinite(v)]
        if r >= vals[-1]:
            s = vals[-1]
        else:
            best = min(range(len(vals)), key=lambda i: (abs(vals[i] - r), i & 1))
            s = vals[best]
        return s if s > 0 else 2.0 ** -9
    raise ValueError(scale)


def _bf_code(q, code):
    if code == "int8":
        r = round(q)                              # Python round is half-even
        return max(-127, min(127, r))
    vals = F.table(code)
    n_mag = len(vals) // 2
    qmax = max(v for v in vals[:n_mag] if math.isfinite(v))
    qc = max(-qmax, min(qmax, q))
    sign = 1 if math.copysign(1, qc) < 0 else 0
    best = None
    for c in range(n_mag):
        if not math.isfinite(vals[c]):
            continue
        key = (abs(abs(qc) - vals[c]), c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1] | (sign << (F.get(code).bits - 1))


def _bf_quantize(x, block, code, scale):
    rows, cols = x.shape
    br, bc = block
    codes = np.zeros((rows, cols), dtype=np.int64)
    scales = np.zeros((rows // br, cols // bc), dtype=np.float64)
    for i in range(rows // br):
        for j in range(cols // bc):
            absmax = 0.0
            for r in range(i * br, (i + 1) * br):
                for c in range(j * bc, (j + 1) * bc):
                    absmax = max(absmax, abs(float(x[r, c])))
            s = _bf_scale(absmax, code, scale)
            scales[i, j] = s
            for r in range(i * br, (i + 1) * br):
                for c in range(j * bc, (j + 1) * bc):
                    codes[r, c] = _bf_code(_r32(float(x[r, c]) / s), code)
    return codes, scales


def _decoded_scales(stored, scale):
    if scale == "f32":
        return np.asarray(stored, np.float64)
    return F.decode(stored, scale)


@pytest.mark.parametrize("code,scale", [("e4m3", "f32"), ("e5m2", "f32"), ("int8", "f32"),
                                        ("e4m3", "ue8m0"), ("e5m2", "ue8m0"), ("e2m1", "ue8m0"),
                                        ("e2m1", "ue4m3"), ("e4m3", "ue4m3")])
@pytest.mark.parametrize("block", [(1, 8), (4, 1), (2, 4)])
def test_quantize_brute_force(code, scale, block):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((8, 16)) * np.exp(rng.uniform(-3, 3, (8, 1)))).astype(np.float32)
    x[1, :] = 0                                   # zero blocks
    x[5, 3] = -0.0
    codes, stored = Q.quantize(x, block, code, scale)
    ref_codes, ref_s = _bf_quantize(x, block, code, scale)
    np.testing.assert_array_equal(_decoded_scales(stored, scale), ref_s)
    if code == "e2m1":
        codes = F.unpack_e2m1(codes)
    if code == "int8":
        np.testing.assert_array_equal(codes.astype(np.int64), ref_codes)
    else:
        np.testing.assert_array_equal(codes.astype(np.int64), ref_codes)


def test_transpose_out_is_transpose():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 96)).astype(np.float32)
    for code in ("e4m3", "e5m2", "e2m1"):
        c, s = Q.quantize(x, (32, 1), code, "ue8m0")
        ct, st = Q.quantize(x, (32, 1), code, "ue8m0", transpose_out=True)
        if code == "e2m1":
            c, ct = F.unpack_e2m1(c), F.unpack_e2m1(ct)
        np.testing.assert_array_equal(ct, c.T)
        np.testing.assert_array_equal(st, s.T)


# ----------------------------------------------------------------------------
# Defining inequalities / invariants
# ----------------------------------------------------------------------------

def test_ue8m0_is_smallest_power_of_two_not_below_ratio():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((256, 64)) * np.exp2(rng.integers(-60, 60, (256, 1)))).astype(np.float32)
    for code, qmax in (("e4m3", 448.0), ("e5m2", 57344.0), ("e2m1", 6.0)):
        amax = Q.block_absmax(x, (1, 32))
        _, stored = Q.block_scales(amax, code, "ue8m0")
        s = F.decode(stored, "ue8m0")
        r = Q.div32(amax, np.float32(qmax)).astype(np.float64)
        assert (s >= r).all() and (s / 2 < r).all()
        # the power of two is exact in binary32 and lies in range
        assert ((stored >= 0) & (stored <= 254)).all()


def test_ue8m0_zero_and_extreme_blocks():
    x = np.zeros((3, 32), np.float32)
    x[1, 0] = 3.4e38
    x[2, 0] = 1e-44                               # ratio underflows to zero
    _, stored = Q.quantize(x, (1, 32), "e4m3", "ue8m0")
    assert stored[0, 0] == 127                   # all-zero block -> scale 1
    assert stored[1, 0] == 127 + 120             # 3.4e38/448 ~ 2**119.6
    assert stored[2, 0] == 0                     # clamped at 2**-127


def test_int8_invariants():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((50, 70)).astype(np.float32)
    x[7] = 0
    q, s = Q.int8_per_row(x)
    assert s[7] == 1.0 and (q[7] == 0).all()
    recon = q.astype(np.float64) * s[:, None]
    err = np.abs(recon - x)
    assert (err <= s[:, None] * (0.5 + 1e-6)).all()
    nz = np.arange(50) != 7
    assert (np.abs(q[nz]).max(axis=1) == 127).all()   # the absmax element hits 127


def test_fp_codes_within_half_step():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 128)).astype(np.float32)
    c, s = Q.quantize(x, (1, 128), "e4m3", "f32")
    deq = Q.dequantize(c, s, (1, 128), "e4m3", "f32")
    # E4M3 normal values carry 3 mantissa bits: relative step 2**-3
    rel = np.abs(deq - x) / np.maximum(np.abs(x), 2.0 ** -6 * np.repeat(s, 128, 1))
    assert (rel <= 2.0 ** -4 + 1e-9).all()


def test_int8_exact_ties_round_half_even():
    """Quotients exactly halfway between integers (absmax 127 makes s = 1):
    rounding goes to the even integer, as jnp.round / Python's round do."""
    x = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5]], np.float32)
    q, s = Q.int8_per_row(x)
    assert s[0] == 1.0
    assert q.tolist() == [[127, 0, 2, 2, 0, -2, -2, 126]]
    assert [round(v) for v in x[0].tolist()] == q[0].tolist()


def test_fp_ties_round_half_even_through_quantizer():
    """A quotient at the midpoint of two E4M3 values takes the even code."""
    x = np.array([[448.0, 1.0625, 1.1875, -1.0625]], np.float32)   # s = 1
    c, s = Q.quantize(x, (1, 4), "e4m3", "f32")
    assert s[0, 0] == 1.0
    assert F.decode(c, "e4m3").tolist() == [[448.0, 1.0, 1.25, -1.0]]


def test_ceil_log2_meets_its_definition():
    """ceil(log2 r) is the integer c with 2^(c-1) < r <= 2^c, checked in exact
    arithmetic on powers of two, their float32 neighbours, subnormals and
    random values over the whole binary32 range."""
    rng = np.random.default_rng(3)
    powers = np.array([2.0 ** e for e in range(-149, 128)], np.float32)
    r = np.concatenate([powers, np.nextafter(powers, np.float32(np.inf)), np.nextafter(powers, np.float32(0)),
                        rng.uniform(1e-3, 1e3, 2000).astype(np.float32),
                        (2.0 ** rng.uniform(-140, 127, 2000)).astype(np.float32)])
    r = r[(r > 0) & np.isfinite(r)]
    c = Q.ceil_log2(r)
    for v, ci in zip(r.tolist(), c.tolist()):
        assert math.ldexp(1.0, ci - 1) < v <= math.ldexp(1.0, ci), (v, ci)


def test_int8_per_column_is_per_row_of_the_transpose():
    """A per-column scale of w is the per-row scale of w^T: codes and scales
    agree element for element (TensorTonic, problem statement)."""
    rng = np.random.default_rng(4)
    w = rng.standard_normal((37, 23)).astype(np.float32)
    w[:, 5] = 0
    qc, sc = Q.int8_per_col(w)
    qr, sr = Q.int8_per_row(w.T.copy())
    np.testing.assert_array_equal(qc, qr.T)
    np.testing.assert_array_equal(sc, sr)
    assert sc[5] == 1.0 and not qc[:, 5].any()


def test_code_values_ties_and_saturation():
    """Quotients on a tie go to the even integer (INT8) and past the format's
    largest value saturate to it (INT8 127, E4M3 448, E5M2 57344, E2M1 6)."""
    q = np.array([2.5, -2.5, 3.5, 0.5, -0.5, 127.6, -300.0], np.float32)
    np.testing.assert_array_equal(Q.code_values(q, "int8"), [2, -2, 4, 0, 0, 127, -127])
    for code, top in (("e4m3", 448.0), ("e5m2", 57344.0), ("e2m1", 6.0)):
        v = F.decode(Q.code_values(np.array([top * 4, -top * 4, top], np.float32), code), code)
        np.testing.assert_array_equal(v, [top, -top, top])
