"""GPU quantizer vs the oracle: codes and scales must be bit-exact.

Inputs are seeded normals with per-row magnitudes spread over e^[-3,3], plus
the degenerate cases of the method: an all-zero row and column, negative
zeros, quotients deep in the subnormal range and one value near the binary32
maximum."""

import zlib

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import quantize as Q

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_x(rows, cols, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.empty(rows, 1).uniform_(-3, 3, generator=g))
    x[1] = 0.0
    x[:, 1] = 0.0
    x[2] *= 1e-36
    x[3, 5] = 3.0e38
    x[4, ::7] = -0.0
    return x.to(DT[dtype])


def oracle_quantize(x, block, code, scale, transpose):
    return Q.quantize(x.float().numpy(), block, code, scale, transpose_out=transpose)


def run_case(rows, cols, block, code, scale, dtype, transpose, seed):
    import block_scaled_precision_gemm_gb300 as bsmm
    x = make_x(rows, cols, seed, dtype)
    codes, scales = bsmm.quantize(x.cuda(), block, code, scale, transpose=transpose)
    torch.cuda.synchronize()
    rc, rs = oracle_quantize(x, block, code, scale, transpose)
    got_c = codes.cpu().numpy()
    if code == "int8":
        got_c = got_c.astype(np.int8)
    np.testing.assert_array_equal(got_c, rc)
    got_s = scales.cpu().numpy()
    if scale == "f32":
        np.testing.assert_array_equal(got_s.view(np.uint32), np.asarray(rs, np.float32).view(np.uint32))
    else:
        np.testing.assert_array_equal(got_s, rs)
    assert bsmm.check_device_status()[0] == 0


FORMATS = [("e4m3", "f32"), ("e5m2", "f32"), ("int8", "f32"), ("e4m3", "ue8m0"), ("e5m2", "ue8m0"),
           ("e2m1", "ue8m0"), ("e2m1", "ue4m3"), ("e4m3", "ue4m3")]


@pytest.mark.parametrize("code,scale", FORMATS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bc", [16, 32, 128])
def test_row_blocks(code, scale, dtype, bc):
    run_case(160, 384, (1, bc), code, scale, dtype, False, seed=bc)


@pytest.mark.parametrize("code,scale", FORMATS)
@pytest.mark.parametrize("br,rows", [(16, 144), (32, 160), (128, 256)])
@pytest.mark.parametrize("transpose", [False, True])
def test_col_blocks(code, scale, br, rows, transpose):
    run_case(rows, 200, (br, 1), code, scale, "bf16" if br == 32 else "f32", transpose, seed=br + rows)


@pytest.mark.parametrize("code,scale", [("e4m3", "f32"), ("e2m1", "ue4m3"), ("e5m2", "ue8m0")])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tile_blocks_128x128(code, scale, dtype):
    run_case(256, 384, (128, 128), code, scale, dtype, False, seed=7)


@pytest.mark.parametrize("code,scale", [("int8", "f32"), ("e4m3", "ue8m0"), ("e2m1", "ue4m3")])
def test_whole_row_and_column_blocks(code, scale):
    run_case(37, 250, (1, 250), code, scale, "f32", False, seed=11)
    run_case(38, 70, (38, 1), code, scale, "f32", False, seed=12)
    run_case(38, 70, (38, 1), code, scale, "f32", True, seed=13)


@pytest.mark.parametrize("block", [(2, 4), (4, 2), (1, 6), (3, 1)])
def test_other_block_shapes(block):
    run_case(12, 24, block, "e4m3", "f32", "f32", False, seed=17)
    if block[1] == 1:
        run_case(12, 24, block, "e5m2", "ue8m0", "f32", True, seed=18)


def test_atrex_recipe_full_width():
    """The block_scaled_mm activation/weight recipe at n = k = 2048 widths."""
    run_case(349, 2048, (1, 128), "e4m3", "f32", "f32", False, seed=21)
    run_case(256, 2048, (128, 128), "e4m3", "f32", "f32", False, seed=22)


def test_empty_input_launches_nothing():
    import block_scaled_precision_gemm_gb300 as bsmm
    x = torch.empty((0, 128), device="cuda")
    c, s = bsmm.quantize(x, (1, 128), "e4m3", "f32")
    assert c.shape == (0, 128) and s.shape == (0, 1)


def test_block_quotient_equals_ieee_division():
    """Every quantizer divides through one correctly rounded reciprocal per
    block and two exact-remainder corrections (Markstein's method) instead of
    a division per element.  On 2 x 2^32 pseudo-random pairs -- divisors with
    random, all-ones and zero significands, quotients on and next to the code
    grids' rounding ties, tiny x -- it must agree bit for bit with the
    hardware's correctly rounded division (bsmm_selftest_quotient)."""
    import block_scaled_precision_gemm_gb300 as bsmm
    for seed in (1, 2**40 + 7):
        assert bsmm.selftest_quotient(1 << 32, seed) == 0


def tie_input(rows, cols, block, code, seed):
    """Blocks whose elements divide by the block's scale onto rounding ties of
    the code grid, or one or two ulps beside them.  Each block holds its
    absmax A once; the scale is s = A / qmax in binary32 (the method's FP32
    scale), and the other elements are RN(m s) nudged by -2..2 ulps, with m a
    midpoint between neighbouring codes (INT8: k + 1/2), so that x / s lands
    within a few ulps of a tie."""
    rng = np.random.default_rng(seed)
    if code == "int8":
        qmax = 127.0
        mids = np.arange(-127, 127) + 0.5
    else:
        v = np.unique(np.abs(F.table(code)[np.isfinite(F.table(code))]))
        mids = (v[:-1] + v[1:]) / 2
        mids = np.concatenate([mids, -mids])
        qmax = F.max_finite(code)
    br, bc = block
    x = np.empty((rows, cols), np.float32)
    for i in range(0, rows, br):
        for j in range(0, cols, bc):
            A = np.float32(np.exp2(rng.uniform(-20, 20)))
            if rng.random() < 0.3:  # an all-ones significand scale
                A = (np.float32(np.exp2(np.floor(rng.uniform(-20, 20)))) * np.float32(2 - 2**-23)).astype(np.float32)
            s = np.float32(A / np.float32(qmax))
            m = rng.choice(mids, size=(br, bc))
            blk = (m * np.float64(s)).astype(np.float32)
            blk = (blk.view(np.int32) + rng.integers(-2, 3, size=blk.shape).astype(np.int32)).view(np.float32)
            blk = np.clip(blk, -A, A)
            blk.flat[rng.integers(0, br * bc)] = A
            x[i:i + br, j:j + bc] = blk
    return torch.from_numpy(x)


@pytest.mark.parametrize("code,block", [("e4m3", (1, 128)), ("e5m2", (1, 128)), ("int8", (1, 128)),
                                        ("e4m3", (128, 128)), ("int8", (128, 128)), ("e4m3", (32, 1)),
                                        ("e4m3", (1, 16))])
def test_quotients_on_rounding_ties(code, block):
    import block_scaled_precision_gemm_gb300 as bsmm
    x = tie_input(256, 512, block, code, seed=zlib.crc32(f"{code}{block}".encode()))
    codes, scales = bsmm.quantize(x.cuda(), block, code, "f32")
    torch.cuda.synchronize()
    rc, rs = oracle_quantize(x, block, code, "f32", False)
    got_c = codes.cpu().numpy()
    if code == "int8":
        got_c = got_c.astype(np.int8)
    np.testing.assert_array_equal(got_c, rc)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), np.asarray(rs, np.float32).view(np.uint32))
    assert bsmm.check_device_status()[0] == 0


@pytest.mark.parametrize("B,D_in,D_out", [(256, 512, 384), (130, 4096, 256), (64, 4224, 128)])
def test_int8_channel_codes_on_rounding_ties(B, D_in, D_out):
    """The INT8 call's own quantizers (x per row, w per column, the latter
    with the rows held in registers up to 4096 and streamed beyond) on
    quotients at and beside k + 1/2."""
    import block_scaled_precision_gemm_gb300 as bsmm
    x = tie_input(B, D_in, (1, D_in), "int8", seed=B + D_in)
    w = tie_input(D_in, D_out, (D_in, 1), "int8", seed=D_in + D_out)
    out = bsmm.int8_channel(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    xq, xs = Q.int8_per_row(x.numpy())
    wq, ws = Q.int8_per_col(w.numpy())
    np.testing.assert_array_equal(out["x_q"].cpu().numpy(), xq)
    np.testing.assert_array_equal(out["w_q"].cpu().numpy(), wq)
    np.testing.assert_array_equal(out["x_scales"].cpu().numpy().view(np.uint32), np.asarray(xs, np.float32).view(np.uint32))
    np.testing.assert_array_equal(out["w_scales"].cpu().numpy().view(np.uint32), np.asarray(ws, np.float32).view(np.uint32))
    assert bsmm.check_device_status()[0] == 0


def test_quantize_batch_matches_the_oracle():
    """bsmm_quantize_batch: 20 jobs of 128 x 128 tiles in one input type and
    scale kind (one launch of 16, one of 4), others of each other kind, and
    jobs on the other quantizers (row blocks, transposed column blocks, a
    zero-sized job) in one call; every job's codes and scales bit-exact."""
    import block_scaled_precision_gemm_gb300 as bsmm
    specs = [(256 + 128 * (i % 3), 384 - 128 * (i % 2), (128, 128), "e4m3", "f32", "f32", False) for i in range(20)]
    specs += [(384, 256, (128, 128), "e2m1", "ue4m3", "bf16", False), (256, 256, (128, 128), "e5m2", "ue8m0", "f32", False),
              (256, 512, (128, 128), "int8", "f32", "bf16", False), (128, 128, (128, 128), "e4m3", "ue8m0", "bf16", False),
              (160, 384, (1, 32), "e4m3", "ue8m0", "f32", False), (144, 200, (16, 1), "e5m2", "ue8m0", "bf16", True)]
    xs = [make_x(r, c, 1000 + i, dt) for i, (r, c, _, _, _, dt, _) in enumerate(specs)]
    jobs = [{"x": x.cuda(), "block": blk, "code": code, "scale": scale, "transpose": tr}
            for x, (_, _, blk, code, scale, _, tr) in zip(xs, specs)]
    jobs.insert(3, {"x": torch.empty(0, 256, device="cuda"), "block": (128, 128)})
    out = bsmm.quantize_batch(jobs)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    del out[3]
    for x, (codes, scales), (_, _, blk, code, scale, _, tr) in zip(xs, out, specs):
        rc, rs = oracle_quantize(x, blk, code, scale, tr)
        got_c = codes.cpu().numpy()
        np.testing.assert_array_equal(got_c.astype(np.int8) if code == "int8" else got_c, rc)
        got_s = scales.cpu().numpy()
        if scale == "f32":
            np.testing.assert_array_equal(got_s.view(np.uint32), np.asarray(rs, np.float32).view(np.uint32))
        else:
            np.testing.assert_array_equal(got_s, rs)
