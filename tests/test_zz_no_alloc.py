"""bsmm_gemm_noalloc: the GEMM entry point for callers that cannot allocate
device memory (for example a plugin inside a framework that owns every
device allocation, or a service that forbids allocations after start-up).
Its scratch is a static device array inside the library.

Each output is checked against the float64 oracle (jax.nn.scaled_matmul,
"Mathematically") and against the allocating entry point, bsmm_gemm, within
the GEMM parity tolerance the other tests use:
|y - y_ref| <= 2e-3 * sum_k |a_s * b_s| per entry.  The calls come two in a
row with different shapes and formats on one stream, with no synchronization
between them: the array keeps the previous call's contents, so the second
call must not depend on them.  Both kernels are forced in turn; the CTA-pair
kernel is the one that writes the skewed and replicated scale blocks into
the array.  This file is named to be collected last."""

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
    """Codes and scales from seeded draws through the oracle's codec, with
    the oracle's product and per-entry bound (float64, per batch)."""
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
    a_s, b_s = G.scaled_operand(da, dsa), G.scaled_operand(db, dsb)
    y_ref = np.stack([a_s[i] @ b_s[i].T for i in range(Bn)])
    bound = np.stack([np.abs(a_s[i]) @ np.abs(b_s[i]).T for i in range(Bn)])
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    return {"a": t(a), "b": t(b), "sa": t(sa), "sb": t(sb), "types": types, "K": K, "shape": (Bn, M, N),
            "y_ref": y_ref, "bound": bound, "what": f"{fmt} {Bn}x{M}x{N}x{K}"}


def _call_noalloc(lib, bsmm, c, y):
    Bn, M, N = c["shape"]
    types = c["types"]
    st = lib.bsmm_gemm_noalloc(Bn, M, N, c["K"], ctypes.c_void_p(c["a"].data_ptr()), bsmm._code(types[0]),
                               ctypes.c_void_p(c["b"].data_ptr()), bsmm._code(types[1]),
                               ctypes.c_void_p(c["sa"].data_ptr()), c["sa"].shape[-1],
                               ctypes.c_void_p(c["sb"].data_ptr()), c["sb"].shape[-1], bsmm._scale(types[2]),
                               ctypes.c_void_p(y.data_ptr()), bsmm.F32,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == bsmm.OK, lib.bsmm_last_error().decode()


def _within(y, y_ref, bound, what):
    ok = G.within_bound(y, y_ref, bound)
    assert ok.all(), f"{what}: {(~ok).sum()} of {ok.size} entries outside 2e-3 * sum|a_s b_s|"


# Pairs of back-to-back calls: different formats, shapes and batch counts.
# The pair-kernel shapes span several 256 x 256 tiles with ragged M and N
# tails; NVFP4 there takes the replicated B blocks.
CALL_PAIRS = {
    "single": [(11, 2, 200, 136, 512, "mxfp8"), (12, 1, 256, 384, 1024, "nvfp4")],
    "pair": [(13, 1, 520, 392, 768, "nvfp4"), (14, 3, 300, 264, 384, "mxfp8")],
}


@pytest.mark.parametrize("kernel", sorted(CALL_PAIRS))
def test_noalloc_gemm_two_calls_in_a_row(monkeypatch, kernel):
    monkeypatch.setenv("BSMM_MX_KERNEL", kernel)
    bsmm, lib = _lib()
    cases = [_mx_case(*spec) for spec in CALL_PAIRS[kernel]]
    ys = [torch.full(c["shape"], float("nan"), dtype=torch.float32, device="cuda") for c in cases]
    for c, y in zip(cases, ys):  # one stream, no synchronization between the calls
        _call_noalloc(lib, bsmm, c, y)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    for c, y in zip(cases, ys):
        y_gemm = bsmm.gemm(c["a"], c["b"], c["sa"], c["sb"], *c["types"], K=c["K"])
        torch.cuda.synchronize()
        yn = y.cpu().numpy()
        assert np.isfinite(yn).all(), c["what"]
        _within(yn, c["y_ref"], c["bound"], f"no-alloc vs oracle, {c['what']}")
        _within(yn, y_gemm.cpu().numpy(), c["bound"], f"no-alloc vs bsmm_gemm, {c['what']}")


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
