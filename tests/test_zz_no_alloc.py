"""bsmm_gemm_noalloc: the GEMM entry point for callers that cannot allocate
device memory (for example a plugin inside a framework that owns every
device allocation, or a service that forbids allocations after start-up).
Its scratch is a static device array inside the library.

Checked against the allocating entry point, bsmm_gemm, on two calls in a row
(the array keeps the previous call's contents, so the second call must not
depend on them), within the GEMM parity tolerance the other tests use:
|y - y_ref| <= 2e-3 * sum_k |a_s * b_s| per entry.  This file is named to be
collected last."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as G

pytestmark = pytest.mark.gpu


def _lib():
    import block_scaled_precision_gemm_gb300 as bsmm
    return bsmm, bsmm.lib()


def _mx_case(seed, Bn, M, N, K, fmt):
    g = torch.Generator().manual_seed(seed)
    if fmt == "mxfp8":
        a = F.encode(torch.randn(Bn, M, K, generator=g).numpy(), "e4m3")
        b = F.encode(torch.randn(Bn, N, K, generator=g).numpy(), "e5m2")
        sa = (torch.randint(-6, 7, (Bn, M, K // 32), generator=g).numpy() + 127).astype(np.uint8)
        sb = (torch.randint(-6, 7, (Bn, N, K // 32), generator=g).numpy() + 127).astype(np.uint8)
        da, db = F.decode(a, "e4m3"), F.decode(b, "e5m2")
        dsa, dsb = F.decode(sa, "ue8m0"), F.decode(sb, "ue8m0")
        types = ("e4m3", "e5m2", "ue8m0")
    else:
        a = torch.randint(0, 256, (Bn, M, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
        b = torch.randint(0, 256, (Bn, N, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
        sa = F.encode(np.exp2(torch.empty(Bn, M, K // 16).uniform_(-4, 4, generator=g).numpy()), "ue4m3")
        sb = F.encode(np.exp2(torch.empty(Bn, N, K // 16).uniform_(-4, 4, generator=g).numpy()), "ue4m3")
        da, db = F.decode(F.unpack_e2m1(a), "e2m1"), F.decode(F.unpack_e2m1(b), "e2m1")
        dsa, dsb = F.decode(sa, "ue4m3"), F.decode(sb, "ue4m3")
        types = ("e2m1", "e2m1", "ue4m3")
    bound = G.scaled_matmul_bound(da, db, dsa, dsb)
    return a, b, sa, sb, types, bound


def _call_noalloc(lib, bsmm, a, b, sa, sb, types, K, y):
    Bn, M = a.shape[0], a.shape[1]
    N = b.shape[1]
    st = lib.bsmm_gemm_noalloc(Bn, M, N, K, ctypes.c_void_p(a.data_ptr()), bsmm._code(types[0]),
                               ctypes.c_void_p(b.data_ptr()), bsmm._code(types[1]),
                               ctypes.c_void_p(sa.data_ptr()), sa.shape[-1], ctypes.c_void_p(sb.data_ptr()),
                               sb.shape[-1], bsmm._scale(types[2]), ctypes.c_void_p(y.data_ptr()), bsmm.F32,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == bsmm.OK, lib.bsmm_last_error().decode()


def test_noalloc_gemm_matches_gemm_on_two_calls_in_a_row():
    bsmm, lib = _lib()
    cases = [(11, 2, 200, 136, 512, "mxfp8"), (12, 1, 256, 384, 1024, "nvfp4")]
    for seed, Bn, M, N, K, fmt in cases:
        a, b, sa, sb, types, bound = _mx_case(seed, Bn, M, N, K, fmt)
        t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
        ta, tb, tsa, tsb = t(a), t(b), t(sa), t(sb)
        y_ref = bsmm.gemm(ta, tb, tsa, tsb, types[0], types[1], types[2], K=K)
        y = torch.full((Bn, M, N), float("nan"), dtype=torch.float32, device="cuda")
        _call_noalloc(lib, bsmm, ta, tb, tsa, tsb, types, K, y)
        torch.cuda.synchronize()
        assert bsmm.check_device_status()[0] == 0
        yn, yr = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(yn).all()
        ok = G.within_bound(yn, yr, bound)
        assert ok.all(), f"{fmt}: {(~ok).sum()} entries differ beyond the tolerance"


def test_noalloc_rejects_problems_beyond_its_scratch():
    bsmm, lib = _lib()
    fake = ctypes.c_void_p(1 << 20)
    # MXFP8, B=8 x 8192 x 8192 x 16384 needs 64 MiB of scale atoms > 32 MiB
    need = lib.bsmm_gemm_workspace_size(8, 8192, 8192, 16384, bsmm.E4M3)
    assert need > bsmm.NOALLOC_SCRATCH_BYTES
    st = lib.bsmm_gemm_noalloc(8, 8192, 8192, 16384, fake, bsmm.E4M3, fake, bsmm.E4M3, fake, 512, fake, 512,
                               bsmm.SCALE_UE8M0, fake, bsmm.F32, None)
    assert st == bsmm.ERR_WORKSPACE
    assert b"at most" in lib.bsmm_last_error()
