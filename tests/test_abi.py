"""The C-ABI library builds, loads and exports every entry point the header
declares; argument validation and the workspace queries run without a GPU
(they return before any CUDA call)."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "bsmm.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import block_scaled_precision_gemm_gb300 as bsmm
    return bsmm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsmm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("bsmm_quantize", "bsmm_gemm", "bsmm_gemm_grouped", "bsmm_int8_channel", "bsmm_linear_backward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_error_string(lib):
    assert lib.bsmm_version() >= 100
    assert isinstance(lib.bsmm_last_error(), bytes)


def test_validation_without_gpu(lib):
    import block_scaled_precision_gemm_gb300 as b
    P = ctypes.c_void_p
    fake = P(4096)
    # K not a multiple of the scale count
    st = lib.bsmm_gemm(1, 128, 128, 100, fake, b.E4M3, fake, b.E4M3, fake, 3, fake, 4, b.SCALE_UE8M0, fake, b.F32,
                       fake, 1 << 20, None)
    assert st == b.ERR_SHAPE
    # the definition takes any block size; what has no kernel: FP8 codes with
    # E2M1 codes, INT8 codes, FP32 scales
    for at, bt, scale in ((b.E4M3, b.E2M1, b.SCALE_UE8M0), (b.INT8, b.INT8, b.SCALE_UE8M0),
                          (b.E4M3, b.E4M3, b.SCALE_F32)):
        st = lib.bsmm_gemm(1, 128, 128, 256, fake, at, fake, bt, fake, 8, fake, 8, scale, fake, b.F32,
                           fake, 1 << 20, None)
        assert st == b.ERR_UNSUPPORTED
        assert b"E4M3/E5M2" in lib.bsmm_last_error()
    # grouped: n not a multiple of group_n; group other than 128
    assert lib.bsmm_gemm_grouped(64, 200, 256, fake, b.E4M3, fake, b.E4M3, fake, fake, 128, 128, fake,
                                 None) == b.ERR_SHAPE
    assert lib.bsmm_gemm_grouped(64, 256, 256, fake, b.E4M3, fake, b.E4M3, fake, fake, 64, 64, fake,
                                 None) == b.ERR_UNSUPPORTED
    # quantize: INT8 needs F32 scales; bad enums; indivisible blocks
    assert lib.bsmm_quantize(fake, b.F32, 4, 32, 32, 1, 32, b.INT8, b.SCALE_UE8M0, 0, fake, 32, fake, 1,
                             None) == b.ERR_UNSUPPORTED
    assert lib.bsmm_quantize(fake, 9, 4, 32, 32, 1, 32, b.E4M3, b.SCALE_F32, 0, fake, 32, fake, 1,
                             None) == b.ERR_INVALID_ARG
    assert lib.bsmm_quantize(fake, b.F32, 4, 33, 33, 1, 32, b.E4M3, b.SCALE_F32, 0, fake, 33, fake, 1,
                             None) == b.ERR_SHAPE
    # zero-sized problems are OK and launch nothing
    assert lib.bsmm_gemm_grouped(0, 256, 256, None, b.E4M3, None, b.E4M3, None, None, 128, 128, None, None) == b.OK
    assert lib.bsmm_gemm(1, 0, 128, 64, None, b.E4M3, None, b.E4M3, None, 2, None, 2, b.SCALE_UE8M0, None, b.F32,
                         None, 0, None) == b.OK
    # missing workspace is reported before any launch
    st = lib.bsmm_gemm(1, 128, 128, 64, fake, b.E4M3, fake, b.E4M3, fake, 2, fake, 2, b.SCALE_UE8M0, fake, b.F32,
                       None, 0, None)
    assert st == b.ERR_WORKSPACE
    # backward needs multiples of 32
    assert lib.bsmm_linear_backward(fake, fake, fake, 33, 64, 64, b.E5M2, fake, fake, fake, 1 << 30,
                                    None) == b.ERR_SHAPE


def test_workspace_queries(lib):
    import block_scaled_precision_gemm_gb300 as b
    # scale slots of 512 B per operand and K tile: the most of the one-CTA
    # layout (atoms per row tile of 128, rounded to pairs) and the pair
    # kernel's blocks (A: atoms + 3 per row tile, one atom as is; NVFP4's B:
    # 8 x atoms per pair of row tiles)
    assert lib.bsmm_gemm_workspace_size(1, 128, 128, 128, b.E4M3) == 2 * (2 * 512)
    assert lib.bsmm_gemm_workspace_size(8, 4096, 4096, 8192, b.E4M3) == 2 * 8 * 32 * 64 * 512
    # E2M1: NVFP4's B blocks, 32 slots per pair of row tiles (room also for MXFP4)
    assert lib.bsmm_gemm_workspace_size(1, 16384, 16384, 16384, b.E2M1) == 2 * 64 * (64 * 32) * 512
    assert lib.bsmm_int8_channel_workspace_size(1, 3, 2) > 0
    assert lib.bsmm_linear_backward_workspace_size(64, 64, 64) > 4 * 64 * 64


def test_atom_layout_queries_and_validation_without_gpu(lib):
    """The tensor-core scale layout entry points: sizes from the documented
    geometry, and argument errors reported before any CUDA call."""
    import block_scaled_precision_gemm_gb300 as b
    P = ctypes.c_void_p
    fake = P(4096)
    # 512-byte atoms [B][ceil(R/256)*2 row tiles][ceil(K/kt) * kt/bs/4 atoms]
    assert lib.bsmm_scale_atoms_size(1, 300, 384, b.E4M3, b.SCALE_UE8M0) == 1 * 4 * 3 * 512
    assert lib.bsmm_scale_atoms_size(2, 256, 1024, b.E5M2, b.SCALE_UE8M0) == 2 * 2 * 8 * 512
    assert lib.bsmm_scale_atoms_size(1, 100, 512, b.E2M1, b.SCALE_UE8M0) == 1 * 2 * (2 * 2) * 512   # MXFP4
    assert lib.bsmm_scale_atoms_size(1, 100, 512, b.E2M1, b.SCALE_UE4M3) == 1 * 2 * (2 * 4) * 512   # NVFP4
    assert lib.bsmm_scale_atoms_size(1, 64, 64, b.E4M3, b.SCALE_UE4M3) == 0  # no tensor-core format
    assert lib.bsmm_scale_atoms_size(1, 64, 64, b.INT8, b.SCALE_F32) == 0
    # quantize to atoms
    q = lib.bsmm_quantize_atoms
    assert q(fake, b.BF16, 1, 64, 64, 0, b.E4M3, b.SCALE_UE4M3, fake, fake, 1 << 20, None) == b.ERR_UNSUPPORTED
    assert q(fake, b.BF16, 1, 64, 48, 0, b.E4M3, b.SCALE_UE8M0, fake, fake, 1 << 20, None) == b.ERR_SHAPE
    assert q(fake, b.BF16, 2, 64, 64, 1, b.E4M3, b.SCALE_UE8M0, fake, fake, 1 << 20, None) == b.ERR_SHAPE
    assert q(fake, b.BF16, 1, 64, 64, 0, b.E4M3, b.SCALE_UE8M0, fake, fake, 100, None) == b.ERR_WORKSPACE
    assert q(fake, b.BF16, 1, 64, 64, 0, b.E4M3, b.SCALE_UE8M0, fake, P(4097), 1 << 20, None) == b.ERR_ALIGNMENT
    assert q(None, b.BF16, 0, 64, 64, 0, b.E4M3, b.SCALE_UE8M0, None, None, 0, None) == b.OK
    # GEMM from atoms: both operands one format; FP4 needs the workspace
    g = lib.bsmm_gemm_atoms
    assert g(1, 128, 128, 256, fake, b.E4M3, fake, b.E2M1, fake, fake, b.SCALE_UE8M0, fake, b.F32, None, 0,
             None) == b.ERR_UNSUPPORTED
    assert g(1, 128, 128, 80, fake, b.E4M3, fake, b.E4M3, fake, fake, b.SCALE_UE8M0, fake, b.F32, None, 0,
             None) == b.ERR_SHAPE
    assert g(1, 128, 128, 256, fake, b.E2M1, fake, b.E2M1, fake, fake, b.SCALE_UE4M3, fake, b.F32, None, 0,
             None) == b.ERR_WORKSPACE
    # pre-quantized backward: multiples of 32; workspace only with row-major scales
    bq = lib.bsmm_linear_backward_quantized
    assert bq(33, 64, 64, b.E5M2, fake, fake, fake, fake, fake, fake, fake, fake, 1, fake, fake, None, 0,
              None) == b.ERR_SHAPE
    assert lib.bsmm_linear_backward_quantized_workspace_size(256, 512, 384, 1) == 0
    assert lib.bsmm_linear_backward_quantized_workspace_size(256, 512, 384, 0) == max(
        lib.bsmm_gemm_workspace_size(1, 256, 384, 512, b.E4M3), lib.bsmm_gemm_workspace_size(1, 512, 384, 256, b.E4M3))
    assert bq(256, 512, 384, b.E5M2, fake, fake, fake, fake, fake, fake, fake, fake, 0, fake, fake, None, 0,
              None) == b.ERR_WORKSPACE


def test_atom_sizes_follow_the_documented_geometry(lib):
    """bsmm_scale_atoms_size over many shapes: 512-byte atoms, [B][ceil(R/256)
    * 2 row tiles][ceil(K/kt) * kt/bs/4 atoms], kt the K of one 128-byte code
    tile (128 for FP8, 256 for E2M1), bs the hardware block (32, or 16 for
    UE4M3); zero for shapes the tensor cores take no scales for."""
    import math
    import random
    import block_scaled_precision_gemm_gb300 as b
    fmts = [(b.E4M3, b.SCALE_UE8M0, 128, 32), (b.E5M2, b.SCALE_UE8M0, 128, 32),
            (b.E2M1, b.SCALE_UE8M0, 256, 32), (b.E2M1, b.SCALE_UE4M3, 256, 16)]
    rnd = random.Random(7)
    for _ in range(300):
        code, scale, kt, bs = rnd.choice(fmts)
        B, R, K = rnd.randint(1, 4), rnd.randint(1, 3000), bs * rnd.randint(1, 200)
        want = B * math.ceil(R / 256) * 2 * math.ceil(K / kt) * (kt // bs // 4) * 512
        assert lib.bsmm_scale_atoms_size(B, R, K, code, scale) == want, (B, R, K, code, scale)
    assert lib.bsmm_scale_atoms_size(0, 64, 64, b.E4M3, b.SCALE_UE8M0) == 0
    assert lib.bsmm_scale_atoms_size(1, 0, 64, b.E4M3, b.SCALE_UE8M0) == 0


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """Without the compiled library every entry point raises: there is no CPU
    or other fallback path."""
    import block_scaled_precision_gemm_gb300 as b
    monkeypatch.setattr(b, "_LIB", None)
    monkeypatch.setattr(b, "library_path", str(tmp_path / "libbsmm.so"))
    with pytest.raises(RuntimeError, match="is missing"):
        b.lib()
    with pytest.raises(RuntimeError, match="is missing"):
        b.gemm_workspace_size(1, 128, 128, 128, "e4m3")
    with pytest.raises(RuntimeError, match="is missing"):
        b.version()


def test_trace_and_selftest_argument_checks_without_gpu(lib):
    """The trace store is host state: start clears it, an empty trace reads
    as out of range, stop leaves it; the quotient self-test refuses a NULL
    counter before any launch."""
    import block_scaled_precision_gemm_gb300 as b
    assert lib.bsmm_trace_start() == b.OK
    assert lib.bsmm_trace_count() == 0
    name, t0, ms = ctypes.c_char_p(), ctypes.c_float(), ctypes.c_float()
    assert lib.bsmm_trace_read(0, ctypes.byref(name), ctypes.byref(t0), ctypes.byref(ms)) == b.ERR_INVALID_ARG
    assert lib.bsmm_trace_read(-1, None, None, None) == b.ERR_INVALID_ARG
    assert lib.bsmm_trace_stop() == b.OK
    assert lib.bsmm_trace_count() == 0
    assert lib.bsmm_selftest_quotient(16, 1, None, None) == b.ERR_INVALID_ARG


def test_quantize_batch_argument_checks_without_gpu(lib):
    """bsmm_quantize_batch checks every job before it launches anything: a
    bad count or jobs pointer, then the first bad job by index; zero jobs and
    zero-sized jobs are no-ops.  The ctypes job matches the C layout (LP64)."""
    import block_scaled_precision_gemm_gb300 as b
    J = b._QuantizeJob
    assert ctypes.sizeof(J) == 96
    assert lib.bsmm_quantize_batch(None, -1, None) == b.ERR_INVALID_ARG
    assert lib.bsmm_quantize_batch(None, 1, None) == b.ERR_INVALID_ARG
    assert lib.bsmm_quantize_batch(None, 0, None) == b.OK
    ok = J(0x1000, b.F32, 256, 256, 256, 128, 128, b.E4M3, b.SCALE_F32, 0, 0x2000, 256, 0x3000, 2)
    empty = J(None, b.F32, 0, 256, 256, 128, 128, b.E4M3, b.SCALE_F32, 0, None, 256, None, 2)
    ragged = J(0x1000, b.F32, 200, 256, 256, 128, 128, b.E4M3, b.SCALE_F32, 0, 0x2000, 256, 0x3000, 2)
    int8_ue8m0 = J(0x1000, b.F32, 256, 256, 256, 1, 32, b.INT8, b.SCALE_UE8M0, 0, 0x2000, 256, 0x3000, 8)
    assert lib.bsmm_quantize_batch((J * 1)(empty), 1, None) == b.OK
    assert lib.bsmm_quantize_batch((J * 3)(ok, empty, ragged), 3, None) == b.ERR_SHAPE
    assert lib.bsmm_last_error().decode().startswith("job 2:")
    assert lib.bsmm_quantize_batch((J * 2)(int8_ue8m0, ragged), 2, None) == b.ERR_UNSUPPORTED
    assert lib.bsmm_last_error().decode().startswith("job 0:")
