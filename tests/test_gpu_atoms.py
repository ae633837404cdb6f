"""Scales in the tensor cores' atom layout (include/bsmm.h, "Scales in the
tensor cores' own layout"; NKI backward page, Parameters: pre-computed scales
and pre-swizzled inputs).

Against the oracle: the atom quantizer's codes are bit-exact with the
oracle's quantizer, and its atoms, read back through the layout the header
documents, hold the oracle's scale bytes (neutral scale in the padding);
GEMMs and the backward fed atoms built from the oracle's scales match the
oracle's float64 products within the parity bound.  Against the row-major
path: the same scales placed by the layout, and the same output bits."""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

FORMATS = {  # name: (code, scale, hardware block, K per 128-byte tile)
    "mxfp8": ("e4m3", "ue8m0", 32, 128),
    "mxfp8_e5m2": ("e5m2", "ue8m0", 32, 128),
    "mxfp4": ("e2m1", "ue8m0", 32, 256),
    "nvfp4": ("e2m1", "ue4m3", 16, 256),
}


def _bsmm():
    import block_scaled_precision_gemm_gb300 as bsmm
    return bsmm


def atoms_from_row_major(sc, B, R, K, fmt):
    """The documented atom layout, written out: row 128 t + w, block 4 j + i
    at byte (w % 32) * 16 + (w / 32) * 4 + i of atom (b, t, j); neutral scale
    elsewhere."""
    _, scale, bs, kt = FORMATS[fmt]
    KS = K // bs
    ks4 = math.ceil(K / kt) * (kt // bs // 4)
    RT = math.ceil(R / 256) * 2
    out = np.full((B, RT, ks4, 512), 0 if scale == "ue4m3" else 127, dtype=np.uint8)
    b, r, kb = np.meshgrid(np.arange(B), np.arange(R), np.arange(KS), indexing="ij")
    t, w = r // 128, r % 128
    j, i = kb // 4, kb % 4
    out[b, t, j, (w % 32) * 16 + (w // 32) * 4 + i] = sc.reshape(B, R, KS)
    return out.reshape(-1)


@pytest.mark.parametrize("fmt", sorted(FORMATS))
@pytest.mark.parametrize("B,R,K,transpose", [(1, 300, 384, False), (2, 130, 256, False), (1, 77, 512, False),
                                             (1, 200, 288, True), (1, 256, 1024, True)])
def test_quantize_atoms_layout(fmt, B, R, K, transpose):
    bsmm = _bsmm()
    code, scale, bs, _ = FORMATS[fmt]
    if K % bs or (code == "e2m1" and K % 2):
        pytest.skip("K must be a multiple of the block")
    g = torch.Generator().manual_seed(B * R + K)
    x = (torch.randn(B * R, K, generator=g) * 3).to(torch.bfloat16).cuda()
    xin = x.t().contiguous() if transpose else x
    codes_a, atoms = bsmm.quantize_atoms(xin, code, scale, batches=B, transpose=transpose)
    if transpose:
        codes_r, sc = bsmm.quantize(xin, (bs, 1), code, scale, transpose=True)
    else:
        codes_r, sc = bsmm.quantize(x, (1, bs), code, scale)
    torch.cuda.synchronize()
    assert torch.equal(codes_a, codes_r)
    want = atoms_from_row_major(sc.cpu().numpy(), B, R, K, fmt)
    assert atoms.numel() == want.size == bsmm.scale_atoms_size(B, R, K, code, scale)
    got = atoms.cpu().numpy()
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} atom bytes differ, first at {bad[:8].tolist()}"


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("fmt", sorted(FORMATS))
@pytest.mark.parametrize("Bn,M,N,K", [(1, 512, 512, 512), (2, 300, 384, 768), (1, 256, 136, 256)])
def test_gemm_atoms_equals_gemm(monkeypatch, kernel, fmt, Bn, M, N, K):
    bsmm = _bsmm()
    code, scale, bs, _ = FORMATS[fmt]
    if fmt == "mxfp4" and kernel == "single":
        pytest.skip("MXFP4 has only the pair kernel")
    monkeypatch.setenv("BSMM_MX_KERNEL", kernel)
    g = torch.Generator().manual_seed(Bn * M + N + K)
    xa = torch.randn(Bn * M, K, generator=g).cuda()
    xb = torch.randn(Bn * N, K, generator=g).cuda()
    ca, sa = bsmm.quantize(xa, (1, bs), code, scale)
    cb, sb = bsmm.quantize(xb, (1, bs), code, scale)
    ka, aa = bsmm.quantize_atoms(xa, code, scale, batches=Bn)
    kb, ab = bsmm.quantize_atoms(xb, code, scale, batches=Bn)
    kd = K // 2 if code == "e2m1" else K
    y_row = bsmm.gemm(ca.view(Bn, M, kd), cb.view(Bn, N, kd), sa.view(Bn, M, -1), sb.view(Bn, N, -1), code, code,
                      scale, K=K)
    y_atm = bsmm.gemm_atoms(ka.view(Bn, M, kd), kb.view(Bn, N, kd), aa, ab, code, code, scale, K=K)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    assert torch.equal(y_row.view(torch.int32), y_atm.view(torch.int32))


@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (512, 256, 256)])
def test_backward_quantized_equals_backward(M, N, K):
    """dX and dW from pre-quantized operands, with row-major and with atom
    scales, equal the backward that quantizes itself."""
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(M + N + K)
    dY = torch.randn(M, N, generator=g).to(torch.bfloat16).cuda()
    W = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    X = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    dX0, dW0 = bsmm.linear_backward(dY, W, X, "e5m2")
    # row-major scales, as bsmm_quantize writes them
    q_dy_n = bsmm.quantize(dY, (1, 32), "e5m2", "ue8m0")
    q_w_t = bsmm.quantize(W, (32, 1), "e5m2", "ue8m0", transpose=True)
    q_dy_t = bsmm.quantize(dY, (32, 1), "e5m2", "ue8m0", transpose=True)
    q_x_t = bsmm.quantize(X, (32, 1), "e5m2", "ue8m0", transpose=True)
    dX1, dW1 = bsmm.linear_backward_quantized(*q_dy_n, *q_w_t, *q_dy_t, *q_x_t, fp8="e5m2")
    # atom scales
    a_dy_n = bsmm.quantize_atoms(dY, "e5m2", "ue8m0")
    a_w_t = bsmm.quantize_atoms(W, "e5m2", "ue8m0", transpose=True)
    a_dy_t = bsmm.quantize_atoms(dY, "e5m2", "ue8m0", transpose=True)
    a_x_t = bsmm.quantize_atoms(X, "e5m2", "ue8m0", transpose=True)
    dX2, dW2 = bsmm.linear_backward_quantized(*a_dy_n, *a_w_t, *a_dy_t, *a_x_t, fp8="e5m2", scales_are_atoms=True)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    for a, b in ((dX0, dX1), (dW0, dW1), (dX0, dX2), (dW0, dW2)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_atoms_reject_other_formats():
    bsmm = _bsmm()
    x = torch.zeros(64, 64, device="cuda")
    assert bsmm.scale_atoms_size(1, 64, 64, "e4m3", "ue4m3") == 0
    with pytest.raises(bsmm.BsmmError):
        bsmm.quantize_atoms(x, "e4m3", "ue4m3")
    with pytest.raises(bsmm.BsmmError):
        bsmm.quantize_atoms(x[:, :48].contiguous(), "e4m3", "ue8m0")  # K not a multiple of 32


# ---------------------------------------------------------------------------
# against the oracle
# ---------------------------------------------------------------------------

from oracle import formats as F  # noqa: E402
from oracle import gemm as G  # noqa: E402
from oracle import quantize as Q  # noqa: E402


def _layout(B, R, K, fmt):
    _, scale, bs, kt = FORMATS[fmt]
    KS = K // bs
    ks4 = math.ceil(K / kt) * (kt // bs // 4)
    RT = math.ceil(R / 256) * 2
    return KS, ks4, RT, (0 if scale == "ue4m3" else 127)


def decode_atoms(atoms, B, R, K, fmt):
    """The header's atom layout read back: scale bytes [B, R, K / bs]; asserts
    that every padding byte holds the neutral scale."""
    KS, ks4, RT, neutral = _layout(B, R, K, fmt)
    a = np.asarray(atoms).reshape(B, RT, ks4, 512)
    r = np.arange(RT * 128)
    kb = np.arange(ks4 * 4)
    byte = ((r % 128) % 32 * 16 + (r % 128) // 32 * 4)[:, None] + (kb % 4)[None, :]
    full = a[:, (r // 128)[:, None], (kb // 4)[None, :], byte]  # [B, RT*128, ks4*4]
    assert (full[:, R:, :] == neutral).all() and (full[:, :, KS:] == neutral).all(), "padding not neutral"
    return full[:, :R, :KS]


def encode_atoms(sc, B, R, K, fmt):
    """Scale bytes [B, R, K / bs] written into the header's atom layout."""
    return atoms_from_row_major(np.asarray(sc, np.uint8), B, R, K, fmt)


@pytest.mark.parametrize("fmt", sorted(FORMATS))
@pytest.mark.parametrize("B,R,K,transpose", [(1, 300, 384, False), (2, 130, 256, False), (1, 200, 288, True),
                                             (1, 256, 1024, True)])
def test_quantize_atoms_matches_oracle(fmt, B, R, K, transpose):
    bsmm = _bsmm()
    code, scale, bs, _ = FORMATS[fmt]
    if K % bs:
        pytest.skip("K must be a multiple of the block")
    g = torch.Generator().manual_seed(7 * B * R + K)
    x = (torch.randn(B * R, K, generator=g) * 3).to(torch.bfloat16)
    xin = x.t().contiguous() if transpose else x
    codes, atoms = bsmm.quantize_atoms(xin.cuda(), code, scale, batches=B, transpose=transpose)
    torch.cuda.synchronize()
    oc, osc = Q.quantize(x.float().numpy(), (1, bs), code, scale)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    got = decode_atoms(atoms.cpu().numpy(), B, R, K, fmt)
    np.testing.assert_array_equal(got, osc.reshape(B, R, -1))


def _oracle_operand(fmt, Bn, R, K, g):
    """Codes and scales by the oracle's quantizer from seeded draws, and the
    scaled float64 operand."""
    code, scale, bs, _ = FORMATS[fmt]
    x = torch.randn(Bn * R, K, generator=g).numpy() * 2
    c, s = Q.quantize(x, (1, bs), code, scale)
    v = F.decode(F.unpack_e2m1(c), "e2m1") if code == "e2m1" else F.decode(c, code)
    return c.reshape(Bn, R, -1), s.reshape(Bn, R, -1), G.scaled_operand(v, F.decode(s, scale)).reshape(Bn, R, K)


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("fmt", sorted(FORMATS))
@pytest.mark.parametrize("Bn,M,N,K", [(1, 512, 512, 512), (2, 300, 384, 768), (3, 600, 520, 256)])
def test_gemm_atoms_matches_oracle(monkeypatch, kernel, fmt, Bn, M, N, K):
    if fmt == "mxfp4" and kernel == "single":
        pytest.skip("MXFP4 has only the pair kernel")
    monkeypatch.setenv("BSMM_MX_KERNEL", kernel)
    bsmm = _bsmm()
    code, scale, _, _ = FORMATS[fmt]
    g = torch.Generator().manual_seed(11 * Bn + M + 3 * N + K)
    ca, sa, a_s = _oracle_operand(fmt, Bn, M, K, g)
    cb, sb, b_s = _oracle_operand(fmt, Bn, N, K, g)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    y = bsmm.gemm_atoms(t(ca), t(cb), t(encode_atoms(sa, Bn, M, K, fmt)), t(encode_atoms(sb, Bn, N, K, fmt)),
                        code, code, scale, K=K)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    y_ref = np.stack([a_s[i] @ b_s[i].T for i in range(Bn)])
    bound = np.stack([np.abs(a_s[i]) @ np.abs(b_s[i]).T for i in range(Bn)])
    ok = G.within_bound(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"{fmt}[{kernel}] {Bn}x{M}x{N}x{K}: {(~ok).sum()} entries outside the bound"


@pytest.mark.parametrize("atoms", [True, False])
@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (512, 256, 256), (1024, 768, 2048)])
def test_backward_quantized_matches_oracle(atoms, M, N, K):
    """dX and dW from operands the oracle quantized along their contraction
    axes (NKI backward, introduction), with row-major or atom scales."""
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(M + 2 * N + K)
    dY = torch.randn(M, N, generator=g).to(torch.bfloat16).float().numpy()
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).float().numpy()
    X = (torch.randn(M, K, generator=g) * 0.02).to(torch.bfloat16).float().numpy()
    ops = {"dy_n": G.mx_quantize(dY, "cols", "e5m2"), "w_t": G.mx_quantize(W, "rows", "e5m2"),
           "dy_t": G.mx_quantize(dY, "rows", "e5m2"), "x_t": G.mx_quantize(X, "rows", "e5m2")}
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    args = []
    for c, s in ops.values():
        R, Kc = c.shape
        args += [t(c), t(encode_atoms(s[None], 1, R, Kc, "mxfp8_e5m2") if atoms else s)]
    dX, dW = bsmm.linear_backward_quantized(*args, fp8="e5m2", scales_are_atoms=atoms)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    op = {k: G.scaled_operand(F.decode(c, "e5m2"), F.decode(s, "ue8m0")) for k, (c, s) in ops.items()}
    for got, a_s, b_s, what in ((dX, op["dy_n"], op["w_t"], "dX"), (dW, op["dy_t"], op["x_t"], "dW")):
        ok = G.within_bound(got.float().cpu().numpy(), a_s @ b_s.T, np.abs(a_s) @ np.abs(b_s).T,
                            out_round=G.BF16_HALF_ULP)
        assert ok.all(), f"{what} (atoms={atoms}): {(~ok).sum()} entries outside the bound"
