"""Element-by-element oracle parity for the CTA-pair GEMMs at sizes with more
256 x 256 output tiles than the GPU has clusters (76 on GB300), so that every
cluster runs several tiles in turn: the persistent tile loop, the reuse of
the tensor-memory buffers across tiles, the barrier phases that flip from one
tile to the next, the output staging ring and the copy warps' prefetch of the
next tile's scales are all on the checked path.  Every output entry is
compared, ragged M and N tails included.

Inputs are seeded draws through the oracle's codec or quantizer; references
are float64, one batch at a time as ``a_s @ b_s.T`` with the scales repeated
along K (the form the oracle's pins tie to the einsum of jax.nn.scaled_matmul,
"Mathematically"), or the oracle's own grouped and backward functions.
Gate: |y - y_ref| <= 2e-3 * sum_k |a_s * b_s| per entry, plus half a bf16 ulp
(2^-8 |y_ref|) for bf16 outputs."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as G
from oracle import quantize as Q

pytestmark = pytest.mark.gpu
REL = 2e-3
CLUSTERS = 76


def _bsmm():
    import block_scaled_precision_gemm_gb300 as bsmm
    return bsmm


def _tiles(Bn, M, N):
    return Bn * -(-M // 256) * -(-N // 256)


def _check(y, y_ref, bound, what, out_round=0.0):
    y = np.asarray(y, np.float64)
    ok = G.within_bound(y, y_ref, bound, REL, out_round)
    if not ok.all():
        idx = np.argwhere(~ok)[:4].tolist()
        raise AssertionError(f"{what}: {(~ok).sum()} of {ok.size} entries outside the bound; first at {idx}")


def _t(v):
    return torch.from_numpy(np.ascontiguousarray(v)).cuda()


def _per_batch(a_s, b_s):
    y = np.stack([a_s[i] @ b_s[i].T for i in range(a_s.shape[0])])
    bound = np.stack([np.abs(a_s[i]) @ np.abs(b_s[i]).T for i in range(a_s.shape[0])])
    return y, bound


# ---------------------------------------------------------------------------
# block_scaled_mm: FP32 scales (atrex-bench #002, Reference Implementation)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("m,n,k", [(8269, 2048, 1024), (4100, 1152, 512), (4100, 1152, 384)])
def test_grouped_pair_several_tiles_per_cluster(monkeypatch, m, n, k):
    """264 and 85 tiles over 76 clusters; m has a tail of 77 and 4 rows, and
    n = 1152 ends in a half-empty tile (n % 256 == 128).  k = 384 gives an
    odd number of K blocks, so a cluster's tiles start on alternating TMEM
    buffers (the epilogue's general loop); even counts take the paired one."""
    assert _tiles(1, m, n) > CLUSTERS
    monkeypatch.setenv("BSMM_GROUPED_KERNEL", "pair")
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(m + n + k)
    ca, sa = Q.quantize(torch.randn(m, k, generator=g).numpy(), (1, 128), "e4m3", "f32")
    cb, sb = Q.quantize(torch.randn(n, k, generator=g).numpy(), (128, 128), "e4m3", "f32")
    y = bsmm.gemm_grouped(_t(ca), _t(cb), _t(sa), _t(sb))
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    da, db = F.decode(ca, "e4m3"), F.decode(cb, "e4m3")
    y_ref = G.grouped_matmul(da, db, sa, sb, 128, 128)
    a_s, b_s = G.grouped_operands(da, db, sa, sb, 128, 128)
    _check(y.cpu().numpy(), y_ref, np.abs(a_s) @ np.abs(b_s).T, f"grouped pair m={m} n={n} k={k}")


# ---------------------------------------------------------------------------
# jax.nn.scaled_matmul with the Blackwell formats (Notes)
# ---------------------------------------------------------------------------

def _mx_codes(fmt, Bn, R, K, g):
    if fmt == "mxfp8":
        c = F.encode(torch.randn(Bn, R, K, generator=g).numpy(), "e4m3")
        s = (torch.randint(-6, 7, (Bn, R, K // 32), generator=g).numpy() + 127).astype(np.uint8)
        return c, s, G.scaled_operand(F.decode(c, "e4m3"), F.decode(s, "ue8m0"))
    c = torch.randint(0, 256, (Bn, R, K // 2), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    v = F.decode(F.unpack_e2m1(c), "e2m1")
    if fmt == "mxfp4":
        s = (torch.randint(-6, 7, (Bn, R, K // 32), generator=g).numpy() + 127).astype(np.uint8)
        return c, s, G.scaled_operand(v, F.decode(s, "ue8m0"))
    s = F.encode(np.exp2(torch.empty(Bn, R, K // 16).uniform_(-4, 4, generator=g).numpy()), "ue4m3")
    return c, s, G.scaled_operand(v, F.decode(s, "ue4m3"))


TYPES = {"mxfp8": ("e4m3", "e4m3", "ue8m0"), "mxfp4": ("e2m1", "e2m1", "ue8m0"),
         "nvfp4": ("e2m1", "e2m1", "ue4m3")}


@pytest.mark.parametrize("fmt,Bn,M,N,K,out", [
    ("mxfp8", 3, 2048, 2048, 1024, torch.float32),
    ("mxfp8", 2, 2050, 2056, 512, torch.bfloat16),
    ("nvfp4", 3, 2048, 2048, 1024, torch.float32),
    ("nvfp4", 1, 2310, 2184, 768, torch.float32),
    ("mxfp4", 3, 2048, 2048, 1024, torch.float32),
    ("mxfp4", 2, 1800, 2312, 512, torch.bfloat16),
])
def test_mx_pair_several_tiles_per_cluster(monkeypatch, fmt, Bn, M, N, K, out):
    """B = 3, M = N = 2048 (192 tiles) and ragged shapes over several batches
    (M, N tails of 2..120 rows; bf16 output)."""
    assert _tiles(Bn, M, N) > CLUSTERS
    monkeypatch.setenv("BSMM_MX_KERNEL", "pair")
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(Bn * M + N + K)
    ca, sa, a_s = _mx_codes(fmt, Bn, M, K, g)
    cb, sb, b_s = _mx_codes(fmt, Bn, N, K, g)
    at, bt, st = TYPES[fmt]
    y = bsmm.gemm(_t(ca), _t(cb), _t(sa), _t(sb), at, bt, st, out_dtype=out, K=K)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    y_ref, bound = _per_batch(a_s, b_s)
    _check(y.float().cpu().numpy(), y_ref, bound, f"{fmt} pair {Bn}x{M}x{N}x{K} {out}",
           G.BF16_HALF_ULP if out == torch.bfloat16 else 0.0)


# ---------------------------------------------------------------------------
# NKI "Matmul MXFP8 Backward Kernel API Reference" (introduction)
# ---------------------------------------------------------------------------

def test_linear_backward_several_tiles_per_cluster():
    """dX [2048, 4096] (128 tiles) and dW [2560, 4096] (160 tiles), both on
    the pair kernel, every entry against the oracle."""
    M, N, K = 2048, 2560, 4096
    assert _tiles(1, M, K) > CLUSTERS and _tiles(1, N, K) > CLUSTERS
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(M + N + K)
    dY = torch.randn(M, N, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    X = (torch.randn(M, K, generator=g) * 0.02).to(torch.bfloat16)
    dX, dW = bsmm.linear_backward(dY.cuda(), W.cuda(), X.cuda(), "e5m2")
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    # the oracle's quantizations along each contraction axis (what its
    # linear_backward does), then the products one BLAS matmul each
    dYf, Wf, Xf = dY.float().numpy(), W.float().numpy(), X.float().numpy()
    op = lambda q: G.scaled_operand(F.decode(q[0], "e5m2"), F.decode(q[1], "ue8m0"))  # noqa: E731
    dy_n, wt = op(G.mx_quantize(dYf, "cols", "e5m2")), op(G.mx_quantize(Wf, "rows", "e5m2"))
    dyt, xt = op(G.mx_quantize(dYf, "rows", "e5m2")), op(G.mx_quantize(Xf, "rows", "e5m2"))
    _check(dX.float().cpu().numpy(), dy_n @ wt.T, np.abs(dy_n) @ np.abs(wt).T, "dX", G.BF16_HALF_ULP)
    _check(dW.float().cpu().numpy(), dyt @ xt.T, np.abs(dyt) @ np.abs(xt).T, "dW", G.BF16_HALF_ULP)
