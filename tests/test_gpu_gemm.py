"""GPU GEMMs vs the oracle on small shapes that span several tiles and ragged
tails.  Inputs (codes and scales) come from the oracle's codec applied to
seeded draws, so the GEMMs are checked independently of the GPU quantizer.
Gate: |y - y_ref| <= 2e-3 * sum_k |a_s * b_s| per entry; bf16 outputs may
additionally move by their own rounding, half a bf16 ulp (2^-8 |y_ref|)."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as G
from oracle import quantize as Q

pytestmark = pytest.mark.gpu
REL = 2e-3


def _bsmm():
    import block_scaled_precision_gemm_gb300 as bsmm
    return bsmm


def assert_within(y, y_ref, bound, what, out_round=0.0):
    y = np.asarray(y, np.float64)
    ok = G.within_bound(y, y_ref, bound, REL, out_round)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {(~ok).sum()}/{ok.size} entries outside the bound; first {idx.tolist()}: "
                             f"y={y[tuple(idx[0])]} ref={y_ref[tuple(idx[0])]} bound={bound[tuple(idx[0])]}")


# ---------------------------------------------------------------------------
# block_scaled_mm: 1x128 activation and 128x128 weight FP32 scales
# ---------------------------------------------------------------------------

def grouped_inputs(m, n, k, seed, code="e4m3"):
    g = torch.Generator().manual_seed(seed)
    a_raw = torch.randn(m, k, generator=g).numpy()
    b_raw = torch.randn(n, k, generator=g).numpy()
    ca, sa = Q.quantize(a_raw, (1, 128), code, "f32")
    cb, sb = Q.quantize(b_raw, (128, 128), code, "f32")
    return ca, sa, cb, sb


def run_grouped(ca, sa, cb, sb, code="e4m3", bcode=None):
    bsmm = _bsmm()
    bcode = bcode or code
    y = bsmm.gemm_grouped(torch.from_numpy(ca).cuda(), torch.from_numpy(cb).cuda(), torch.from_numpy(sa).cuda(),
                          torch.from_numpy(sb).cuda(), 128, 128, a_type=code, b_type=bcode)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    da, db = F.decode(ca, code), F.decode(cb, bcode)
    y_ref = G.grouped_matmul(da, db, sa, sb, 128, 128)
    a_s, b_s = G.grouped_operands(da, db, sa, sb, 128, 128)
    return y.cpu().numpy(), y_ref, np.abs(a_s) @ np.abs(b_s).T


@pytest.mark.parametrize("m,n,k", [(64, 256, 256), (1, 128, 128), (237, 256, 384), (349, 384, 256),
                                   (300, 640, 1024), (129, 128, 2048)])
def test_grouped_parity(m, n, k):
    y, y_ref, bound = run_grouped(*grouped_inputs(m, n, k, seed=m + n + k))
    assert_within(y, y_ref, bound, f"grouped m={m} n={n} k={k}")


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("m,n,k", [(256, 256, 128), (300, 384, 512), (1, 256, 256), (777, 1024, 1024),
                                   (2000, 2048, 2048)])
def test_grouped_parity_each_kernel(monkeypatch, kernel, m, n, k):
    """Both GEMM kernels (CTA-pair 256x256 tiles and single-CTA 128x128
    tiles) on ragged shapes: an M tail, N % 256 == 128 (a half-empty pair
    tile), a single row, and several waves of tiles."""
    monkeypatch.setenv("BSMM_GROUPED_KERNEL", kernel)
    y, y_ref, bound = run_grouped(*grouped_inputs(m, n, k, seed=3 * m + n))
    assert_within(y, y_ref, bound, f"grouped[{kernel}] m={m} n={n} k={k}")


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("m,n,k", [(349, 256, 2048), (237, 384, 1280), (64, 128, 640)])
def test_grouped_split_k(monkeypatch, splits, m, n, k):
    """Split K on the one-CTA FP32-scale kernel (a cluster of `splits` CTAs
    per tile; each 32 x 64 block's partials summed by one rank, in a fixed
    order, through distributed shared memory), including splits that do not
    divide the K tiles evenly."""
    monkeypatch.setenv("BSMM_GROUPED_KERNEL", "single")
    monkeypatch.setenv("BSMM_GROUPED_SPLITK", str(splits))
    y, y_ref, bound = run_grouped(*grouped_inputs(m, n, k, seed=m + 7 * splits))
    assert_within(y, y_ref, bound, f"split-K {splits}: m={m} n={n} k={k}")


def test_grouped_split_k_is_deterministic(monkeypatch):
    """The split partials are added in a fixed order: repeated calls give
    identical bits."""
    monkeypatch.setenv("BSMM_GROUPED_KERNEL", "single")
    monkeypatch.setenv("BSMM_GROUPED_SPLITK", "4")
    ca, sa, cb, sb = grouped_inputs(300, 256, 2048, seed=5)
    bsmm = _bsmm()
    args = [torch.from_numpy(v).cuda() for v in (ca, cb, sa, sb)]
    y1 = bsmm.gemm_grouped(*args, 128, 128)
    y2 = bsmm.gemm_grouped(*args, 128, 128)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("m,n", [(349, 2048), (237, 4096)])
def test_grouped_small_m_sweep_shapes(m, n):
    """The Shapes-table problems with fewer 128 x 128 tiles than SMs take
    split K by default; full size, checked against the oracle on sampled
    rows."""
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(m)
    a_raw = torch.randn(m, n, generator=g).numpy()
    b_raw = torch.randn(n, n, generator=g).numpy()
    ca, sa = Q.quantize(a_raw, (1, 128), "e4m3", "f32")
    cb, sb = Q.quantize(b_raw, (128, 128), "e4m3", "f32")
    y = bsmm.gemm_grouped(torch.from_numpy(ca).cuda(), torch.from_numpy(cb).cuda(), torch.from_numpy(sa).cuda(),
                          torch.from_numpy(sb).cuda(), 128, 128).cpu().numpy()
    rows = np.array([0, 1, m // 2, m - 1])
    da, db = F.decode(ca[rows], "e4m3"), F.decode(cb, "e4m3")
    y_ref = G.grouped_matmul(da, db, sa[rows], sb, 128, 128)
    a_s, b_s = G.grouped_operands(da, db, sa[rows], sb, 128, 128)
    assert_within(y[rows], y_ref, np.abs(a_s) @ np.abs(b_s).T, f"small-m sweep shape m={m} n=k={n}")


def test_grouped_e5m2_operands():
    ca, sa, _, _ = grouped_inputs(100, 256, 256, 5, "e5m2")
    _, _, cb, sb = grouped_inputs(100, 256, 256, 6, "e4m3")
    y, y_ref, bound = run_grouped(ca, sa, cb, sb, "e5m2", "e4m3")
    assert_within(y, y_ref, bound, "grouped e5m2 x e4m3")


def test_grouped_one_hot_scales():
    """Only one (row, K block) scale and one (n group, K block) scale are
    nonzero: pins the scale indexing of the promotion epilogue."""
    m, n, k = 256, 384, 512
    ca, sa, cb, sb = grouped_inputs(m, n, k, 9)
    sa = np.zeros_like(sa)
    sb = np.zeros_like(sb)
    for r in range(m):
        sa[r, r % 4] = 1.0 + r / 1000
    sb[1, 2] = 0.5
    sb[2, 3] = 2.0
    y, y_ref, bound = run_grouped(ca, sa, cb, sb)
    assert_within(y, y_ref, bound, "one-hot scales")
    assert np.count_nonzero(y_ref) > 0 and (y[:, :128] == 0).all()


def test_grouped_end_to_end_with_gpu_quantizer():
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(3)
    a_raw = torch.randn(237, 1024, generator=g)
    b_raw = torch.randn(512, 1024, generator=g)
    aq, sa = bsmm.quantize(a_raw.cuda(), (1, 128), "e4m3", "f32")
    bq, sb = bsmm.quantize(b_raw.cuda(), (128, 128), "e4m3", "f32")
    y = bsmm.gemm_grouped(aq, bq, sa, sb).cpu().numpy()
    ca, osa = Q.quantize(a_raw.numpy(), (1, 128), "e4m3", "f32")
    cb, osb = Q.quantize(b_raw.numpy(), (128, 128), "e4m3", "f32")
    np.testing.assert_array_equal(aq.cpu().numpy(), ca)
    np.testing.assert_array_equal(bq.cpu().numpy(), cb)
    da, db = F.decode(ca, "e4m3"), F.decode(cb, "e4m3")
    a_s, b_s = G.grouped_operands(da, db, osa, osb, 128, 128)
    assert_within(y, G.grouped_matmul(da, db, osa, osb, 128, 128), np.abs(a_s) @ np.abs(b_s).T, "end to end")


# ---------------------------------------------------------------------------
# batched MXFP8 / NVFP4 (jax.nn.scaled_matmul with the Blackwell formats)
# ---------------------------------------------------------------------------

def mx_inputs(Bn, M, N, K, at, bt, seed, pattern="random"):
    g = torch.Generator().manual_seed(seed)
    ca = F.encode(torch.randn(Bn, M, K, generator=g).numpy(), at)
    cb = F.encode(torch.randn(Bn, N, K, generator=g).numpy(), bt)
    ea = torch.randint(-6, 7, (Bn, M, K // 32), generator=g).numpy()
    eb = torch.randint(-6, 7, (Bn, N, K // 32), generator=g).numpy()
    if pattern == "one_hot_a":     # row m keeps only K block (m % KS); others ~2^-127
        ks = K // 32
        ea = np.full_like(ea, -127)
        for r in range(M):
            ea[:, r, r % ks] = (r % 5) - 2
    elif pattern == "one_hot_b":
        ks = K // 32
        eb = np.full_like(eb, -127)
        for r in range(N):
            eb[:, r, (3 * r + 1) % ks] = (r % 3) - 1
    return ca, cb, (ea + 127).astype(np.uint8), (eb + 127).astype(np.uint8)


def run_mx(Bn, M, N, K, at, bt, out, seed, pattern="random"):
    bsmm = _bsmm()
    ca, cb, sa, sb = mx_inputs(Bn, M, N, K, at, bt, seed, pattern)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    y = bsmm.gemm(t(ca), t(cb), t(sa), t(sb), at, bt, "ue8m0", out_dtype=out)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    da, db = F.decode(ca, at), F.decode(cb, bt)
    dsa, dsb = F.decode(sa, "ue8m0"), F.decode(sb, "ue8m0")
    y_ref = G.scaled_matmul(da, db, dsa, dsb)
    bound = G.scaled_matmul_bound(da, db, dsa, dsb)
    assert_within(y.float().cpu().numpy(), y_ref, bound, f"mxfp8 {Bn}x{M}x{N}x{K} {at}x{bt} {out} {pattern}",
                  G.BF16_HALF_ULP if out == torch.bfloat16 else 0.0)
    return y


@pytest.mark.parametrize("Bn,M,N,K", [(1, 128, 128, 128), (2, 200, 136, 256), (1, 64, 256, 96),
                                      (3, 130, 250, 512), (1, 300, 384, 1024)])
def test_mxfp8_parity(Bn, M, N, K):
    run_mx(Bn, M, N, K, "e4m3", "e4m3", torch.float32, seed=M + N + K)


@pytest.mark.parametrize("at,bt", [("e5m2", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e5m2")])
def test_mxfp8_mixed_formats(at, bt):
    run_mx(2, 160, 192, 256, at, bt, torch.float32, seed=31)


@pytest.mark.parametrize("N", [136, 250])
def test_mxfp8_bf16_output(N):
    """bf16 output = round-to-nearest-even of the same product in FP32, bit
    for bit, and within the bound plus bf16's own half-ulp rounding."""
    y16 = run_mx(2, 200, N, 512, "e5m2", "e5m2", torch.bfloat16, seed=N)
    y32 = run_mx(2, 200, N, 512, "e5m2", "e5m2", torch.float32, seed=N)
    assert torch.equal(y16.cpu().view(torch.int16), y32.cpu().to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("pattern", ["one_hot_a", "one_hot_b"])
def test_mxfp8_scale_layout_one_hot(pattern):
    run_mx(1, 256, 256, 512, "e4m3", "e4m3", torch.float32, seed=41, pattern=pattern)


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("Bn,M,N,K,at,bt,out,pattern", [
    (1, 256, 256, 128, "e4m3", "e4m3", torch.float32, "random"),
    (2, 300, 384, 512, "e4m3", "e4m3", torch.float32, "random"),
    (1, 64, 256, 96, "e4m3", "e4m3", torch.float32, "random"),
    (3, 130, 136, 256, "e5m2", "e4m3", torch.float32, "random"),
    (2, 520, 264, 384, "e4m3", "e5m2", torch.bfloat16, "random"),
    (1, 1, 512, 256, "e4m3", "e4m3", torch.bfloat16, "random"),
    (1, 512, 512, 1024, "e4m3", "e4m3", torch.float32, "one_hot_a"),
    (1, 512, 512, 1024, "e4m3", "e4m3", torch.float32, "one_hot_b"),
])
def test_mxfp8_each_kernel(monkeypatch, kernel, Bn, M, N, K, at, bt, out, pattern):
    """The CTA-pair (256 x 256 tiles) and one-CTA (128 x 128) kernels, each
    forced, on ragged M/N/K, batches, both FP8 formats, bf16 output and
    one-hot scale layouts (a misplaced scale byte selects the wrong block)."""
    monkeypatch.setenv("BSMM_MX_KERNEL", kernel)
    run_mx(Bn, M, N, K, at, bt, out, seed=7 * M + N + K, pattern=pattern)


def nv_inputs(Bn, M, N, K, seed, pattern="random"):
    g = torch.Generator().manual_seed(seed)
    a = torch.randint(0, 256, (Bn, M, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    b = torch.randint(0, 256, (Bn, N, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    sa_v = np.exp2(torch.empty(Bn, M, K // 16).uniform_(-4, 4, generator=g).numpy())
    sb_v = np.exp2(torch.empty(Bn, N, K // 16).uniform_(-4, 4, generator=g).numpy())
    sa, sb = F.encode(sa_v, "ue4m3"), F.encode(sb_v, "ue4m3")
    if pattern == "one_hot_a":
        ks = K // 16
        sa = np.zeros_like(sa)
        for r in range(M):
            sa[:, r, (r * 7) % ks] = 0x38
    return a, b, sa, sb


@pytest.mark.parametrize("Bn,M,N,K,pattern", [(1, 128, 128, 256, "random"), (2, 200, 136, 512, "random"),
                                              (1, 64, 128, 64, "random"), (1, 256, 384, 1024, "random"),
                                              (1, 256, 256, 512, "one_hot_a")])
def test_nvfp4_parity(Bn, M, N, K, pattern):
    bsmm = _bsmm()
    a, b, sa, sb = nv_inputs(Bn, M, N, K, seed=M + K, pattern=pattern)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    y = bsmm.gemm(t(a), t(b), t(sa), t(sb), "e2m1", "e2m1", "ue4m3")
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    da, db = F.decode(F.unpack_e2m1(a), "e2m1"), F.decode(F.unpack_e2m1(b), "e2m1")
    dsa, dsb = F.decode(sa, "ue4m3"), F.decode(sb, "ue4m3")
    y_ref = G.scaled_matmul(da, db, dsa, dsb)
    bound = G.scaled_matmul_bound(da, db, dsa, dsb)
    assert_within(y.cpu().numpy(), y_ref, bound, f"nvfp4 {Bn}x{M}x{N}x{K} {pattern}")


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("Bn,M,N,K,pattern", [(1, 256, 256, 256, "random"), (2, 200, 136, 512, "random"),
                                              (1, 64, 128, 64, "random"), (3, 300, 520, 768, "random"),
                                              (1, 512, 384, 1024, "one_hot_a")])
def test_nvfp4_each_kernel(monkeypatch, kernel, Bn, M, N, K, pattern):
    monkeypatch.setenv("BSMM_MX_KERNEL", kernel)
    test_nvfp4_parity(Bn, M, N, K, pattern)


def test_jax_basic_case_padded_to_a_hardware_block():
    """[1,2,3].[4,5,6] with both scales 0.5 is 8: padded with zero codes to
    K = 32 (one UE8M0 block, scale 2^-1)."""
    bsmm = _bsmm()
    a = np.zeros((1, 1, 32), np.float32); a[0, 0, :3] = [1, 2, 3]
    b = np.zeros((1, 1, 32), np.float32); b[0, 0, :3] = [4, 5, 6]
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    s = np.full((1, 1, 1), 126, np.uint8)
    y = bsmm.gemm(t(F.encode(a, "e4m3")), t(F.encode(b, "e4m3")), t(s), t(s), "e4m3", "e4m3", "ue8m0")
    assert y.cpu().item() == 8.0


def test_jax_cudnn_example_shapes_block_16_ue8m0():
    """The jax cuDNN example's shapes: a, b (3, 128, 64) FP8 with (3, 128, 4)
    E8M0 scales, i.e. a block of 16, which the tensor cores do not scale by:
    computed by the CUDA-core kernel, checked against the definition."""
    run_blocks(3, 128, 128, 64, "e4m3", "e4m3", "ue8m0", 16, 16, seed=64)


def run_blocks(Bn, M, N, K, at, bt, scale, bs_a, bs_b, seed, out=torch.float32):
    """Any block sizes: codes from seeded draws through the oracle's codec,
    scale bytes drawn over a range of the scale format."""
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(seed)

    def codes(rows, fmt):
        if fmt == "e2m1":
            return torch.randint(0, 256, (Bn, rows, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
        return F.encode(torch.randn(Bn, rows, K, generator=g).numpy(), fmt)

    def scales(rows, bs):
        if scale == "ue8m0":
            return (torch.randint(-6, 7, (Bn, rows, K // bs), generator=g).numpy() + 127).astype(np.uint8)
        return F.encode(np.exp2(torch.empty(Bn, rows, K // bs).uniform_(-4, 4, generator=g).numpy()), "ue4m3")

    ca, cb, sa, sb = codes(M, at), codes(N, bt), scales(M, bs_a), scales(N, bs_b)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    y = bsmm.gemm(t(ca), t(cb), t(sa), t(sb), at, bt, scale, out_dtype=out)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    dec = lambda c, f: F.decode(F.unpack_e2m1(c), "e2m1") if f == "e2m1" else F.decode(c, f)  # noqa: E731
    da, db = dec(ca, at), dec(cb, bt)
    dsa, dsb = F.decode(sa, scale), F.decode(sb, scale)
    y_ref = G.scaled_matmul(da, db, dsa, dsb)
    bound = G.scaled_matmul_bound(da, db, dsa, dsb)
    assert_within(y.float().cpu().numpy(), y_ref, bound, f"{at}x{bt} {scale} blocks {bs_a}/{bs_b} {Bn}x{M}x{N}x{K}",
                  G.BF16_HALF_ULP if out == torch.bfloat16 else 0.0)


@pytest.mark.parametrize("at,bt,scale,bs_a,bs_b,K", [
    # multiples of the hardware block: tensor cores, each scale repeated
    ("e4m3", "e4m3", "ue8m0", 64, 64, 512), ("e4m3", "e5m2", "ue8m0", 128, 32, 512),
    ("e2m1", "e2m1", "ue4m3", 32, 64, 512), ("e2m1", "e2m1", "ue8m0", 64, 128, 1024),
    # other blocks: CUDA-core kernel
    ("e4m3", "e4m3", "ue8m0", 16, 16, 256), ("e5m2", "e4m3", "ue8m0", 48, 96, 96),
    ("e4m3", "e4m3", "ue4m3", 32, 32, 256), ("e2m1", "e2m1", "ue8m0", 16, 16, 256),
    ("e2m1", "e2m1", "ue4m3", 8, 8, 64), ("e4m3", "e4m3", "ue8m0", 200, 200, 200),
])
def test_any_block_size(at, bt, scale, bs_a, bs_b, K):
    run_blocks(2, 200, 136, K, at, bt, scale, bs_a, bs_b, seed=bs_a * 7 + bs_b + K)


def test_any_block_size_bf16_output():
    run_blocks(1, 256, 256, 256, "e4m3", "e4m3", "ue8m0", 16, 16, seed=5, out=torch.bfloat16)


@pytest.mark.parametrize("offset", [1, 4])
def test_mxfp8_scales_at_unaligned_base(offset):
    """Scale arrays whose base is not 16-byte aligned (a view into a larger
    buffer) take the relayout's byte path and give the same result."""
    bsmm = _bsmm()
    Bn, M, N, K = 1, 256, 256, 1024
    ca, cb, sa, sb = mx_inputs(Bn, M, N, K, "e4m3", "e4m3", seed=77)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    big_a = torch.zeros(sa.size + offset, dtype=torch.uint8, device="cuda")
    big_b = torch.zeros(sb.size + offset, dtype=torch.uint8, device="cuda")
    va = big_a[offset:].view(sa.shape)
    vb = big_b[offset:].view(sb.shape)
    va.copy_(t(sa))
    vb.copy_(t(sb))
    y = bsmm.gemm(t(ca), t(cb), va, vb, "e4m3", "e4m3", "ue8m0")
    y_ref = bsmm.gemm(t(ca), t(cb), t(sa), t(sb), "e4m3", "e4m3", "ue8m0")
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))


@pytest.mark.parametrize("m,n", [(0, 256), (128, 0)])
def test_grouped_empty_output_is_a_no_op(m, n):
    """An empty M or N gives an empty y and launches nothing (K stays 256)."""
    bsmm = _bsmm()
    a = torch.zeros((m, 256), dtype=torch.uint8, device="cuda")
    b = torch.zeros((n, 256), dtype=torch.uint8, device="cuda")
    sa = torch.ones((m, 2), dtype=torch.float32, device="cuda")
    sb = torch.ones((max(1, (n + 127) // 128), 2), dtype=torch.float32, device="cuda")
    y = bsmm.gemm_grouped(a, b, sa, sb)
    torch.cuda.synchronize()
    assert y.shape == (m, n) and bsmm.check_device_status()[0] == 0


@pytest.mark.parametrize("Bn,M,N", [(0, 64, 64), (2, 0, 64), (2, 64, 0)])
def test_batched_empty_output_is_a_no_op(Bn, M, N):
    bsmm = _bsmm()
    a = torch.zeros((Bn, M, 64), dtype=torch.uint8, device="cuda")
    b = torch.zeros((Bn, N, 64), dtype=torch.uint8, device="cuda")
    sa = torch.full((Bn, M, 2), 127, dtype=torch.uint8, device="cuda")
    sb = torch.full((Bn, N, 2), 127, dtype=torch.uint8, device="cuda")
    y = bsmm.gemm(a, b, sa, sb, "e4m3", "e4m3", "ue8m0")
    torch.cuda.synchronize()
    assert y.shape == (Bn, M, N) and bsmm.check_device_status()[0] == 0


# ---------------------------------------------------------------------------
# MXFP4: E2M1 codes with a UE8M0 scale per 32 elements (jax.nn.scaled_matmul's
# definition with the OCP MX block of 32; CTA-pair kernel only)
# ---------------------------------------------------------------------------

def mxf4_inputs(Bn, M, N, K, seed, pattern="random"):
    g = torch.Generator().manual_seed(seed)
    a = torch.randint(0, 256, (Bn, M, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    b = torch.randint(0, 256, (Bn, N, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    ea = torch.randint(-6, 7, (Bn, M, K // 32), generator=g).numpy()
    eb = torch.randint(-6, 7, (Bn, N, K // 32), generator=g).numpy()
    ks = K // 32
    if pattern == "one_hot_a":  # row m keeps only K block (5m+1) % ks
        ea = np.full_like(ea, -127)
        for r in range(M):
            ea[:, r, (5 * r + 1) % ks] = (r % 5) - 2
    elif pattern == "one_hot_b":
        eb = np.full_like(eb, -127)
        for r in range(N):
            eb[:, r, (3 * r + 2) % ks] = (r % 3) - 1
    return a, b, (ea + 127).astype(np.uint8), (eb + 127).astype(np.uint8)


@pytest.mark.parametrize("Bn,M,N,K,out,pattern", [
    (1, 256, 256, 256, torch.float32, "random"),
    (2, 200, 136, 512, torch.float32, "random"),
    (1, 512, 384, 1024, torch.float32, "random"),
    (3, 300, 520, 768, torch.bfloat16, "random"),
    (1, 1, 256, 96, torch.float32, "random"),
    (1, 512, 512, 1024, torch.float32, "one_hot_a"),
    (1, 512, 512, 1024, torch.float32, "one_hot_b"),
])
def test_mxfp4_parity(Bn, M, N, K, out, pattern):
    bsmm = _bsmm()
    a, b, sa, sb = mxf4_inputs(Bn, M, N, K, seed=M + N + K, pattern=pattern)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()  # noqa: E731
    y = bsmm.gemm(t(a), t(b), t(sa), t(sb), "e2m1", "e2m1", "ue8m0", out_dtype=out)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    da, db = F.decode(F.unpack_e2m1(a), "e2m1"), F.decode(F.unpack_e2m1(b), "e2m1")
    dsa, dsb = F.decode(sa, "ue8m0"), F.decode(sb, "ue8m0")
    y_ref = G.scaled_matmul(da, db, dsa, dsb)
    bound = G.scaled_matmul_bound(da, db, dsa, dsb)
    assert_within(y.float().cpu().numpy(), y_ref, bound, f"mxfp4 {Bn}x{M}x{N}x{K} {pattern}",
                  G.BF16_HALF_ULP if out == torch.bfloat16 else 0.0)
