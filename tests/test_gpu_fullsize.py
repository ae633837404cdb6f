"""Parity at the full benchmark sizes, in the launch configuration bench.py
times: each test builds bench.py's workload object, runs one step through the
C ABI, and checks outputs against the oracle computed from the seeded raw
inputs (rows and columns copied from the generator's output; nothing the
library produced feeds the oracle).

Sampling, per output matrix: 256 rows and 256 columns drawn at random give
256 x 256 = 65,536 random entries, and the first and last 256 rows and
columns are added, so that the four corner 256 x 256 tiles -- the ragged M
tail among them -- are checked in full.  The reference for the whole grid of
sampled rows x sampled columns is one float64 product of the oracle's scaled
operands (``a_s[rows] @ b_s[cols].T``, the form its pins tie to the einsum of
jax.nn.scaled_matmul, "Mathematically").  Codes and scales of the sampled
lines are checked bit-exact; outputs against |y - y_ref| <= 2e-3 *
sum_k |a_s * b_s| (plus half a bf16 ulp for bf16 outputs).  The INT8
configuration is checked in full: every code, scale and output."""

import gc

import numpy as np
import pytest
import torch

import bench
import workloads as W
from oracle import formats as F
from oracle import gemm as G
from oracle import quantize as Q

pytestmark = pytest.mark.gpu
REL = 2e-3
TILE = 256
N_RANDOM = 256


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _check(y, y_ref, bound, what, out_round=0.0):
    ok = G.within_bound(y, y_ref, bound, REL, out_round)
    if not ok.all():
        idx = np.argwhere(~ok)[:4].tolist()
        raise AssertionError(f"{what}: {(~ok).sum()} of {ok.size} sampled entries outside the bound; first {idx}")


def grid_lines(n, rng):
    """N_RANDOM random lines of n, plus the first and the last TILE lines."""
    rand = rng.choice(n, size=min(N_RANDOM, n), replace=False)
    first = np.arange(min(TILE, n))
    last = np.arange((n - 1) // TILE * TILE, n)
    return np.unique(np.concatenate([rand, first, last]))


def _rows(t, idx, device):
    return t[torch.from_numpy(idx).to(device)]


def _grid(t2d, rows, cols, device):
    return t2d[torch.from_numpy(rows).to(device)][:, torch.from_numpy(cols).to(device)]


@pytest.fixture(scope="module")
def device():
    import block_scaled_precision_gemm_gb300 as bsmm
    bsmm.lib()
    return torch.device("cuda", 0)


def test_grid_lines_cover_the_plan():
    rng = np.random.default_rng(0)
    for n in (237, 349, 4533, 704512):
        lines = grid_lines(n, rng)
        assert {0, n - 1} <= set(lines.tolist())
        assert set(range((n - 1) // TILE * TILE, n)) <= set(lines.tolist())
        assert lines.size >= min(n, N_RANDOM)


def test_block_scaled_mm_sweep_sampled(device):
    """All eight Shapes-table problems, one bench step (quantize a, quantize
    b, FP32-scale GEMM)."""
    import block_scaled_precision_gemm_gb300 as bsmm
    wl = bench.GroupedWork(W.GROUPED_SWEEP, device)
    wl.step()
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    rng = np.random.default_rng(0)
    for it in wl.items:
        p = it["p"]
        rows, cols = grid_lines(p.m, rng), grid_lines(p.n, rng)
        # activations: the sampled rows, quantized per 1 x 128
        ca, sa = Q.quantize(_rows(it["a_raw"], rows, device).cpu().numpy(), (1, p.group_k), "e4m3", "f32")
        np.testing.assert_array_equal(_rows(it["aq"], rows, device).cpu().numpy(), ca)
        np.testing.assert_array_equal(_rows(it["sa"], rows, device).cpu().numpy(), sa)
        # weights: whole 128-row groups holding the sampled columns
        b_s = np.empty((cols.size, p.k))
        for g in np.unique(cols // p.group_n):
            blk = it["b_raw"][g * p.group_n:(g + 1) * p.group_n].cpu().numpy()
            cb, sb = Q.quantize(blk, (p.group_n, p.group_k), "e4m3", "f32")
            np.testing.assert_array_equal(it["bq"][g * p.group_n:(g + 1) * p.group_n].cpu().numpy(), cb)
            np.testing.assert_array_equal(it["sb"][g].cpu().numpy(), sb[0])
            sel = np.flatnonzero(cols // p.group_n == g)
            b_s[sel] = G.scaled_operand(F.decode(cb[cols[sel] % p.group_n], "e4m3"), np.repeat(sb, sel.size, 0))
        a_s = G.scaled_operand(F.decode(ca, "e4m3"), sa)
        got = _grid(it["y"], rows, cols, device).cpu().numpy()
        _check(got, a_s @ b_s.T, np.abs(a_s) @ np.abs(b_s).T, f"block_scaled_mm m={p.m} n={p.n} k={p.k}")
    del wl
    _free()


def test_int8_per_channel_full(device):
    """B = D_in = D_out = 4096 with zeroed rows/columns, checked in full:
    codes and scales bit-exact, the integer sums exact (a float64 product of
    integer codes is exact below 2^53), y within 1e-6 of acc * s_x * s_w, and
    a zero sum gives exactly 0."""
    wl = bench.Int8Work(W.INT8_4096, device)
    wl.step()
    torch.cuda.synchronize()
    x, w = wl.x.cpu().numpy(), wl.wt.cpu().numpy()
    x_q, x_s = Q.int8_per_row(x)
    w_q, w_s = Q.int8_per_col(w)
    np.testing.assert_array_equal(wl.out["x_q"].cpu().numpy(), x_q)
    np.testing.assert_array_equal(wl.out["w_q"].cpu().numpy(), w_q)
    np.testing.assert_array_equal(wl.out["x_scales"].cpu().numpy(), x_s)
    np.testing.assert_array_equal(wl.out["w_scales"].cpu().numpy(), w_s)
    acc = x_q.astype(np.float64) @ w_q.astype(np.float64)
    y_ref = acc * x_s.astype(np.float64)[:, None] * w_s.astype(np.float64)[None, :]
    y = wl.out["y"].cpu().numpy().astype(np.float64)
    bad = np.abs(y - y_ref) > 1e-6 * np.abs(y_ref)
    assert not bad.any(), f"{bad.sum()} entries beyond 1e-6 relative"
    assert (y[acc == 0] == 0).all()
    zero_rows = W.zero_lines(wl.p.B, wl.p.zero_frac, W.INT8_4096.seed, W.S_ZERO_ROWS).numpy()
    assert (wl.out["x_scales"].cpu().numpy()[zero_rows] == 1.0).all()
    del wl
    _free()


@pytest.mark.parametrize("workload", [W.MXFP8_BATCHED, W.NVFP4_SQUARE, W.MXFP4_SQUARE],
                         ids=["mxfp8", "nvfp4", "mxfp4"])
def test_batched_scaled_matmul_sampled(device, workload):
    """MXFP8 B=8 x 4096 x 4096 x 8192, NVFP4 and MXFP4 16384^3, one bench
    step; the first, the last and one random batch."""
    import block_scaled_precision_gemm_gb300 as bsmm
    wl = bench.MxWork(workload, device)
    wl.step()
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    p = wl.p
    rng = np.random.default_rng(2)
    fmt = p.fmt
    code = "e4m3" if fmt == "mxfp8" else "e2m1"
    scale = "ue4m3" if fmt == "nvfp4" else "ue8m0"

    def operand(codes, scales, idx):
        c, s = _rows(codes, idx, device).cpu().numpy(), _rows(scales, idx, device).cpu().numpy()
        v = F.decode(c, code) if code == "e4m3" else F.decode(F.unpack_e2m1(c), "e2m1")
        return G.scaled_operand(v, F.decode(s, scale))

    for b in np.unique([0, p.B - 1, rng.integers(0, p.B)]):
        rows, cols = grid_lines(p.M, rng), grid_lines(p.N, rng)
        a_s, b_s = operand(wl.a[b], wl.sa[b], rows), operand(wl.b[b], wl.sb[b], cols)
        got = _grid(wl.y[b], rows, cols, device).cpu().numpy()
        _check(got, a_s @ b_s.T, np.abs(a_s) @ np.abs(b_s).T, f"{workload.name} batch {b}")
    del wl
    _free()


def test_linear_backward_sampled(device):
    """M=16384, N=K=8192 bf16: grids of dX and dW, each from the lines of dY,
    W and X it contracts, quantized by the oracle along its own contraction
    axis."""
    import block_scaled_precision_gemm_gb300 as bsmm
    wl = bench.BackwardWork(W.BACKWARD, device)
    wl.step()
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    p = wl.p
    rng = np.random.default_rng(3)
    fp8 = p.fp8

    def q_rows(v):  # contraction along the rows' own axis, blocks of 32
        c, s = Q.quantize(v, (1, 32), fp8, "ue8m0")
        return G.scaled_operand(F.decode(c, fp8), F.decode(s, "ue8m0"))

    def q_cols(v):  # contraction down the columns: the transposed operand
        c, s = Q.quantize(v, (32, 1), fp8, "ue8m0", transpose_out=True)
        return G.scaled_operand(F.decode(c, fp8), F.decode(s, "ue8m0"))

    # dX [M, K] = dY [M, N] . W [N, K]
    ms, ks = grid_lines(p.M, rng), grid_lines(p.K, rng)
    dy = q_rows(_rows(wl.dY, ms, device).float().cpu().numpy())
    wt = q_cols(wl.W[:, torch.from_numpy(ks).to(device)].float().cpu().numpy())
    _check(_grid(wl.dX, ms, ks, device).float().cpu().numpy(), dy @ wt.T, np.abs(dy) @ np.abs(wt).T, "dX",
           G.BF16_HALF_ULP)
    # dW [N, K] = dY^T [N, M] . X [M, K]
    ns, ks = grid_lines(p.N, rng), grid_lines(p.K, rng)
    dyt = q_cols(wl.dY[:, torch.from_numpy(ns).to(device)].float().cpu().numpy())
    xt = q_cols(wl.X[:, torch.from_numpy(ks).to(device)].float().cpu().numpy())
    _check(_grid(wl.dW, ns, ks, device).float().cpu().numpy(), dyt @ xt.T, np.abs(dyt) @ np.abs(xt).T, "dW",
           G.BF16_HALF_ULP)
    del wl
    _free()


def test_e2e_pipelined_chunks_match_the_plain_step(device, monkeypatch):
    """bench.py's end-to-end step splits each problem into row chunks over
    three streams; every output row depends on its own row alone, so the
    results must equal the plain step's bit for bit.  (Split K, chosen by a
    call's tile count, changes the order of the FP32 sums; it is held at one
    split here because these chunks are far smaller than the Shapes-table
    problems, whose 65536-row chunks all run on the CTA-pair kernel.)"""
    monkeypatch.setenv("BSMM_GROUPED_SPLITK", "1")
    wl_spec = W.Workload("chunked e2e check", 5, (W.Grouped(1000, 256, 384), W.Grouped(3000, 512, 256)))
    wl = bench.GroupedWork(wl_spec, device)
    wl.E2E_ROWS = 256
    wl.setup_host()
    # the host input buffer holds the largest problem's raw inputs; give every
    # problem those values so the two runs see the same data
    for it in wl.items:
        na, nb = it["a_raw"].numel(), it["b_raw"].numel()
        it["a_raw"].view(-1).copy_(wl.hb_in[:na])
        it["b_raw"].view(-1).copy_(wl.hb_in[na:na + nb])
    wl.step()
    torch.cuda.synchronize()
    ref = [it["y"].clone() for it in wl.items]
    for it in wl.items:
        it["y"].zero_()
    wl.step_e2e()
    torch.cuda.synchronize()
    for it, r in zip(wl.items, ref):
        diff = (it["y"].view(torch.int32) != r.view(torch.int32)).sum().item()
        assert diff == 0, f"m={it['p'].m} n={it['p'].n} k={it['p'].k}: {diff} entries differ"
    del wl
    _free()
