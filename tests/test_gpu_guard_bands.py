"""Guard bands around every output: no store lands outside the buffer it
belongs to.  (The GPU memory checker is not available on this machine, so
out-of-bounds stores are caught this way instead.)

Each output, and each workspace, is the interior of a larger device buffer
whose margins -- 1 MiB before and after -- are filled with a sentinel byte.
After a call on a ragged shape the margins must still hold the sentinel.  The
shapes put stores at the edges the kernels special-case: M tails that end
inside a 128- or 256-row tile, N % 256 == 128 (the CTA-pair kernel's
half-empty tile), N not a multiple of 16, D_out not a multiple of 4 or 16
(INT8 through TMA and through the warp-level fallback), quantizer blocks
that end a tile early, and transposed outputs.  Results are checked for
finiteness only; parity is the other tests' job."""

import numpy as np
import pytest
import torch

from oracle import formats as F

pytestmark = pytest.mark.gpu
MARGIN = 1 << 20
SENTINEL = 0xA5


def _bsmm():
    import block_scaled_precision_gemm_gb300 as bsmm
    return bsmm


class Guarded:
    """A tensor of `shape` and `dtype` inside a sentinel-filled buffer."""

    def __init__(self, shape, dtype, fill=None):
        self.nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((2 * MARGIN + self.nbytes,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.buf[MARGIN:MARGIN + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self, what):
        torch.cuda.synchronize()
        head, tail = self.buf[:MARGIN], self.buf[MARGIN + self.nbytes:]
        nh, nt = int((head != SENTINEL).sum()), int((tail != SENTINEL).sum())
        assert nh == 0 and nt == 0, f"{what}: {nh} bytes written before and {nt} after the buffer"


def _status_ok():
    assert _bsmm().check_device_status()[0] == 0


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("m,n,k", [(300, 384, 512), (777, 1152, 256), (2000, 2176, 384), (1, 128, 128)])
def test_grouped_gemm_stays_inside_y(monkeypatch, kernel, m, n, k):
    monkeypatch.setenv("BSMM_GROUPED_KERNEL", kernel)
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(m + n + k)
    a = F.encode(torch.randn(m, k, generator=g).numpy(), "e4m3")
    b = F.encode(torch.randn(n, k, generator=g).numpy(), "e4m3")
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    sa = torch.rand(m, k // 128, generator=g).cuda() + 0.5
    sb = torch.rand(n // 128, k // 128, generator=g).cuda() + 0.5
    y = Guarded((m, n), torch.float32)
    bsmm.gemm_grouped(t(a), t(b), sa, sb, y=y.t)
    y.check(f"grouped[{kernel}] m={m} n={n} k={k}")
    _status_ok()
    assert torch.isfinite(y.t).all()


@pytest.mark.parametrize("rows,cols,block,code,scale,transpose", [
    (300, 384, (1, 128), "e4m3", "f32", False),
    (384, 256, (128, 128), "e4m3", "f32", False),
    (130, 96, (1, 32), "e5m2", "ue8m0", False),
    (160, 200, (32, 1), "e5m2", "ue8m0", True),
    (144, 200, (16, 1), "e2m1", "ue4m3", True),
    (77, 4100, (1, 4100), "int8", "f32", False),
    (4100, 36, (4100, 1), "int8", "f32", False),
])
def test_quantizer_stays_inside_codes_and_scales(rows, cols, block, code, scale, transpose):
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(rows * 7 + cols)
    x = (torch.randn(rows, cols, generator=g) * 3).cuda()
    orows, ocols = (cols, rows) if transpose else (rows, cols)
    width = ocols // 2 if code == "e2m1" else ocols
    srows, scols = (cols // block[1], rows // block[0]) if transpose else (rows // block[0], cols // block[1])
    codes = Guarded((orows, width), torch.int8 if code == "int8" else torch.uint8)
    scales = Guarded((srows, scols), torch.float32 if scale == "f32" else torch.uint8)
    bsmm.quantize(x, block, code, scale, transpose=transpose, codes=codes.t, scales=scales.t)
    codes.check("codes")
    scales.check("scales")
    _status_ok()


def _mx_operands(fmt, Bn, R, K, g):
    if fmt == "mxfp8":
        c = F.encode(torch.randn(Bn, R, K, generator=g).numpy(), "e4m3")
        s = (torch.randint(-4, 5, (Bn, R, K // 32), generator=g).numpy() + 127).astype(np.uint8)
    else:
        c = torch.randint(0, 256, (Bn, R, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
        if fmt == "mxfp4":
            s = (torch.randint(-4, 5, (Bn, R, K // 32), generator=g).numpy() + 127).astype(np.uint8)
        else:
            s = F.encode(np.exp2(torch.empty(Bn, R, K // 16).uniform_(-3, 3, generator=g).numpy()), "ue4m3")
    return torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()


TYPES = {"mxfp8": ("e4m3", "e4m3", "ue8m0"), "mxfp4": ("e2m1", "e2m1", "ue8m0"),
         "nvfp4": ("e2m1", "e2m1", "ue4m3")}


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("fmt,Bn,M,N,K,out", [
    ("mxfp8", 2, 300, 136, 512, torch.float32), ("mxfp8", 3, 130, 392, 256, torch.bfloat16),
    ("mxfp8", 1, 520, 264, 384, torch.float32), ("nvfp4", 1, 520, 392, 768, torch.float32),
    ("nvfp4", 2, 200, 136, 512, torch.float32), ("mxfp4", 2, 200, 264, 256, torch.float32),
    ("mxfp4", 1, 300, 520, 512, torch.bfloat16),
])
def test_mx_gemm_stays_inside_y_and_workspace(monkeypatch, kernel, fmt, Bn, M, N, K, out):
    if fmt == "mxfp4" and kernel == "single":
        pytest.skip("MXFP4 has only the pair kernel")
    monkeypatch.setenv("BSMM_MX_KERNEL", kernel)
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(Bn * M + N + K)
    a, sa = _mx_operands(fmt, Bn, M, K, g)
    b, sb = _mx_operands(fmt, Bn, N, K, g)
    at, bt, sc = TYPES[fmt]
    y = Guarded((Bn, M, N), out)
    ws = Guarded((max(1, bsmm.gemm_workspace_size(Bn, M, N, K, at)),), torch.uint8)
    bsmm.gemm(a, b, sa, sb, at, bt, sc, out_dtype=out, y=y.t, workspace=ws.t, K=K)
    y.check(f"{fmt}[{kernel}] y")
    ws.check(f"{fmt}[{kernel}] workspace")
    _status_ok()
    assert torch.isfinite(y.t.float()).all()


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_noalloc_gemm_stays_inside_y(monkeypatch, kernel):
    monkeypatch.setenv("BSMM_MX_KERNEL", kernel)
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(5)
    a, sa = _mx_operands("nvfp4", 1, 520, 768, g)
    b, sb = _mx_operands("nvfp4", 1, 392, 768, g)
    y = Guarded((1, 520, 392), torch.float32)
    bsmm.gemm_noalloc(a, b, sa, sb, "e2m1", "e2m1", "ue4m3", y=y.t, K=768)
    y.check(f"no-alloc[{kernel}] y")
    _status_ok()


@pytest.mark.parametrize("Bn,D_in,D_out", [(300, 200, 100), (300, 200, 102), (77, 130, 36), (520, 384, 264)])
def test_int8_stays_inside_its_outputs(Bn, D_in, D_out):
    """D_out = 102 is not a multiple of 4: the warp-level integer MMA path;
    the others go through the tensor cores and TMA stores."""
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(Bn + D_in + D_out)
    x = torch.randn(Bn, D_in, generator=g).cuda()
    w = torch.randn(D_in, D_out, generator=g).cuda()
    outs = {"x_q": Guarded((Bn, D_in), torch.int8), "x_scales": Guarded((Bn,), torch.float32),
            "w_q": Guarded((D_in, D_out), torch.int8), "w_scales": Guarded((D_out,), torch.float32),
            "y": Guarded((Bn, D_out), torch.float32), "acc": Guarded((Bn, D_out), torch.int32)}
    ws = Guarded((bsmm.int8_channel_workspace_size(Bn, D_in, D_out),), torch.uint8)
    bsmm.int8_channel(x, w, return_acc=True, out={k: v.t for k, v in outs.items()}, workspace=ws.t)
    for k, v in outs.items():
        v.check(f"int8 {k}")
    ws.check("int8 workspace")
    _status_ok()


@pytest.mark.parametrize("M,N,K", [(160, 96, 224), (288, 416, 160)])
def test_backward_stays_inside_dx_dw_and_workspace(M, N, K):
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(M + N + K)
    dY = torch.randn(M, N, generator=g).to(torch.bfloat16).cuda()
    Wt = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    X = (torch.randn(M, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    dX, dW = Guarded((M, K), torch.bfloat16), Guarded((N, K), torch.bfloat16)
    ws = Guarded((bsmm.linear_backward_workspace_size(M, N, K),), torch.uint8)
    bsmm.linear_backward(dY, Wt, X, "e5m2", dX=dX.t, dW=dW.t, workspace=ws.t)
    dX.check("dX")
    dW.check("dW")
    ws.check("backward workspace")
    _status_ok()


@pytest.mark.parametrize("code,scale,R,K,transpose", [("e4m3", "ue8m0", 300, 384, False),
                                                      ("e2m1", "ue4m3", 130, 512, False),
                                                      ("e5m2", "ue8m0", 200, 288, True)])
def test_quantize_atoms_stays_inside_codes_and_atoms(code, scale, R, K, transpose):
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(R + K)
    x = torch.randn(R, K, generator=g).to(torch.bfloat16).cuda()
    xin = x.t().contiguous() if transpose else x
    codes = Guarded((R, K // 2 if code == "e2m1" else K), torch.uint8)
    atoms = Guarded((bsmm.scale_atoms_size(1, R, K, code, scale),), torch.uint8)
    bsmm.quantize_atoms(xin, code, scale, transpose=transpose, codes=codes.t, atoms=atoms.t)
    codes.check("atom quantizer codes")
    atoms.check("atom quantizer atoms")
    _status_ok()
