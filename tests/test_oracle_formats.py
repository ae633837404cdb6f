"""Pins of the oracle's codecs to things other than the oracle itself:
the OCP format anchors, torch's own float8 conversions (an independent
library), and brute-force nearest search."""

import math
import struct

import numpy as np
import pytest
import torch

from oracle import formats as F


def test_anchor_values_e4m3():
    t = F.table("e4m3")
    assert t[0x7E] == 448.0                       # largest finite
    assert t[0x08] == 2.0 ** -6                   # smallest normal
    assert t[0x01] == 2.0 ** -9                   # smallest subnormal
    assert t[0x38] == 1.0
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2                 # no infinities, two NaNs
    assert t[0x80] == 0.0 and math.copysign(1, t[0x80]) == -1
    assert F.max_finite("e4m3") == 448.0


def test_anchor_values_e5m2():
    t = F.table("e5m2")
    assert t[0x7B] == 57344.0
    assert t[0x7C] == math.inf and t[0xFC] == -math.inf
    assert t[0x01] == 2.0 ** -16 and t[0x04] == 2.0 ** -14
    assert t[0x3C] == 1.0
    assert np.isnan(t).sum() == 6
    assert F.max_finite("e5m2") == 57344.0


def test_anchor_values_e2m1_ue8m0_ue4m3():
    assert list(F.table("e2m1")[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(F.table("e2m1")[8:]) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    u = F.table("ue8m0")
    assert u[127] == 1.0 and u[0] == 2.0 ** -127 and u[254] == 2.0 ** 127
    assert math.isnan(u[255])
    np.testing.assert_array_equal(F.table("ue4m3"), F.table("e4m3")[:128])


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2),
                                     ("ue8m0", torch.float8_e8m0fnu)])
def test_decode_matches_torch(fmt, tdt):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(tdt).to(torch.float64).numpy()
    got = F.decode(codes.numpy(), fmt)
    np.testing.assert_array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ref[ok], got[ok])


def _midpoints_and_neighbours(fmt):
    """Every finite value, every midpoint between neighbours, and the binary32
    neighbours of each midpoint, both signs."""
    _, vals = F._positive_finite(F.get(fmt))
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(0))
    pts = np.concatenate([pts, up, dn])
    return np.concatenate([pts, -pts])


@pytest.mark.parametrize("fmt,tdt,lim", [("e4m3", torch.float8_e4m3fn, 448.0),
                                         ("e5m2", torch.float8_e5m2, 57344.0)])
def test_encode_matches_torch(fmt, tdt, lim):
    rng = np.random.default_rng(0)
    rnd = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 1.0, 30.0, lim / 4)])
    v = np.concatenate([_midpoints_and_neighbours(fmt), rnd]).astype(np.float32)
    v = v[np.abs(v) <= lim]                       # torch does not saturate
    ref = torch.from_numpy(v).to(tdt).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F.encode(v, fmt), ref)


def test_encode_ue4m3_matches_torch_on_positive():
    v = np.abs(_midpoints_and_neighbours("e4m3"))
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F.encode(v, "ue4m3"), ref)


def test_encode_e2m1_brute_force():
    """Nearest of the 16 E2M1 values by exhaustive distance; ties to the even
    code; saturation; sign kept."""
    grid = np.concatenate([np.linspace(-8, 8, 6401), _midpoints_and_neighbours("e2m1"),
                           [0.25, -0.25, 5.0, -5.0, 7.0, 100.0]]).astype(np.float32)
    vals = F.table("e2m1")
    for x in grid:
        x = float(x)
        best = None
        for c in range(16):
            if (c >> 3) != (1 if math.copysign(1, x) < 0 else 0):
                continue                          # sign is carried, not rounded
            d = abs(abs(x) - abs(vals[c])) if abs(x) <= 6 else abs(6 - abs(vals[c]))
            key = (d, c & 1)
            if best is None or key < best[0]:
                best = (key, c)
        assert F.encode(np.float32(x), "e2m1") == best[1], x


def test_roundtrip_every_code():
    for fmt in ("e4m3", "e5m2", "e2m1", "ue4m3"):
        t = F.table(fmt)
        codes = np.arange(len(t))
        ok = np.isfinite(t)
        np.testing.assert_array_equal(F.encode(t[ok].astype(np.float32), fmt), codes[ok])


def test_e2m1_packing_nibble_order():
    packed = F.pack_e2m1(np.array([[1, 2, 3, 4]], dtype=np.uint8))
    assert packed.tolist() == [[0x21, 0x43]]      # even element in the low nibble
    np.testing.assert_array_equal(F.unpack_e2m1(packed), [[1, 2, 3, 4]])


def test_bf16_decode_matches_torch():
    x = torch.randn(1000).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(F.bf16_bits_to_f32(bits), x.float().numpy())


def test_float32_struct_agrees():
    # binary32 interpretation used by the brute-force quantizer tests
    assert struct.unpack("f", struct.pack("f", 0.1))[0] == float(np.float32(0.1))
