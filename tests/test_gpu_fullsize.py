"""Parity at the full benchmark sizes, in the launch configuration bench.py
times: each test builds bench.py's workload object, runs one step through the
C ABI, and checks sampled outputs against the oracle computed one entry at a
time from the seeded raw inputs (rows/columns copied from the generator's
output; nothing the library produced feeds the oracle).  Codes and scales of
the sampled lines are checked bit-exact; outputs against the parity bound."""

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
N_SAMPLES = 48


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _check(y, y_ref, bound, what, out_round=0.0):
    ok = G.within_bound(y, y_ref, bound, REL, out_round)
    assert ok.all(), f"{what}: {(~ok).sum()} of {ok.size} sampled entries outside the bound"


def _rng(seed):
    return np.random.default_rng(seed)


@pytest.fixture(scope="module")
def device():
    import block_scaled_precision_gemm_gb300 as bsmm
    bsmm.lib()
    return torch.device("cuda", 0)


def test_block_scaled_mm_sweep_sampled(device):
    """All eight Shapes-table problems, one bench step (quantize a, quantize
    b, FP32-scale GEMM), ragged M tails included."""
    import block_scaled_precision_gemm_gb300 as bsmm
    wl = bench.GroupedWork(W.GROUPED_SWEEP, device)
    wl.step()
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    rng = _rng(0)
    for it in wl.items:
        p = it["p"]
        rows = np.unique(np.concatenate([rng.integers(0, p.m, N_SAMPLES), [0, p.m - 1]]))
        cols = rng.integers(0, p.n, rows.size)
        groups = np.unique(cols // p.group_n)
        # activations: the sampled rows, quantized per 1 x 128
        a_rows = it["a_raw"][torch.from_numpy(rows).to(device)].cpu().numpy()
        ca, sa = Q.quantize(a_rows, (1, p.group_k), "e4m3", "f32")
        np.testing.assert_array_equal(it["aq"][torch.from_numpy(rows).to(device)].cpu().numpy(), ca)
        np.testing.assert_array_equal(it["sa"][torch.from_numpy(rows).to(device)].cpu().numpy(), sa)
        # weights: whole 128-row groups holding the sampled columns
        b_rows = {}
        for g in groups:
            blk = it["b_raw"][g * p.group_n:(g + 1) * p.group_n].cpu().numpy()
            cb, sb = Q.quantize(blk, (p.group_n, p.group_k), "e4m3", "f32")
            np.testing.assert_array_equal(it["bq"][g * p.group_n:(g + 1) * p.group_n].cpu().numpy(), cb)
            np.testing.assert_array_equal(it["sb"][g].cpu().numpy(), sb[0])
            b_rows[g] = (cb, sb)
        got = it["y"][torch.from_numpy(rows).to(device), torch.from_numpy(cols).to(device)].cpu().numpy()
        da = F.decode(ca, "e4m3")
        db = np.stack([F.decode(b_rows[c // p.group_n][0][c % p.group_n], "e4m3") for c in cols])
        sbs = np.stack([b_rows[c // p.group_n][1][0] for c in cols])
        a_s = G.scaled_operand(da, sa)
        b_s = G.scaled_operand(db, sbs)
        y_ref = (a_s * b_s).sum(-1)
        bound = np.abs(a_s * b_s).sum(-1)
        _check(got, y_ref, bound, f"block_scaled_mm m={p.m} n={p.n} k={p.k}")
    del wl
    _free()


def test_int8_per_channel_sampled(device):
    """B = D_in = D_out = 4096 with zeroed rows/columns; y within 1e-6 of
    acc*sx*sw from exact integer sums; codes and scales bit-exact."""
    wl = bench.Int8Work(W.INT8_4096, device)
    wl.step()
    torch.cuda.synchronize()
    rng = _rng(1)
    p = wl.p
    zero_rows = W.zero_lines(p.B, p.zero_frac, W.INT8_4096.seed, W.S_ZERO_ROWS).numpy()
    bs = np.concatenate([rng.integers(0, p.B, N_SAMPLES), zero_rows[:2]])
    js = rng.integers(0, p.D_out, bs.size)
    for b, j in zip(bs, js):
        x = wl.x[b:b + 1].cpu().numpy()
        w = wl.wt[:, j:j + 1].cpu().numpy()
        ref = G.int8_channel(x, w)
        np.testing.assert_array_equal(wl.out["x_q"][b].cpu().numpy(), ref["x_q"][0])
        np.testing.assert_array_equal(wl.out["w_q"][:, j].cpu().numpy(), ref["w_q"][:, 0])
        assert wl.out["x_scales"][b].item() == ref["x_scales"][0]
        assert wl.out["w_scales"][j].item() == ref["w_scales"][0]
        y = wl.out["y"][b, j].item()
        yr = ref["y_ref"][0, 0]
        assert abs(y - yr) <= 1e-6 * abs(yr), (b, j, y, yr)
        if ref["acc"][0, 0] == 0:
            assert y == 0.0
    del wl
    _free()


@pytest.mark.parametrize("workload", [W.MXFP8_BATCHED, W.NVFP4_SQUARE, W.MXFP4_SQUARE],
                         ids=["mxfp8", "nvfp4", "mxfp4"])
def test_batched_scaled_matmul_sampled(device, workload):
    """MXFP8 B=8 x 4096 x 4096 x 8192, NVFP4 and MXFP4 16384^3, one bench step."""
    import block_scaled_precision_gemm_gb300 as bsmm
    wl = bench.MxWork(workload, device)
    wl.step()
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    p = wl.p
    rng = _rng(2)
    ib = rng.integers(0, p.B, N_SAMPLES)
    im = np.concatenate([rng.integers(0, p.M, N_SAMPLES - 2), [0, p.M - 1]])
    inn = np.concatenate([rng.integers(0, p.N, N_SAMPLES - 2), [p.N - 1, 0]])
    idx_a = (torch.from_numpy(ib).to(device), torch.from_numpy(im).to(device))
    idx_b = (torch.from_numpy(ib).to(device), torch.from_numpy(inn).to(device))
    a, b = wl.a[idx_a].cpu().numpy(), wl.b[idx_b].cpu().numpy()
    sa, sb = wl.sa[idx_a].cpu().numpy(), wl.sb[idx_b].cpu().numpy()
    if p.fmt == "mxfp8":
        da, db = F.decode(a, "e4m3"), F.decode(b, "e4m3")
        dsa, dsb = F.decode(sa, "ue8m0"), F.decode(sb, "ue8m0")
    elif p.fmt == "mxfp4":
        da, db = F.decode(F.unpack_e2m1(a), "e2m1"), F.decode(F.unpack_e2m1(b), "e2m1")
        dsa, dsb = F.decode(sa, "ue8m0"), F.decode(sb, "ue8m0")
    else:
        da, db = F.decode(F.unpack_e2m1(a), "e2m1"), F.decode(F.unpack_e2m1(b), "e2m1")
        dsa, dsb = F.decode(sa, "ue4m3"), F.decode(sb, "ue4m3")
    a_s, b_s = G.scaled_operand(da, dsa), G.scaled_operand(db, dsb)
    y_ref = (a_s * b_s).sum(-1)
    bound = np.abs(a_s * b_s).sum(-1)
    y = wl.y[(idx_a[0], idx_a[1], torch.from_numpy(inn).to(device))].cpu().numpy()
    _check(y, y_ref, bound, workload.name)
    del wl
    _free()


def test_linear_backward_sampled(device):
    """M=16384, N=K=8192 bf16: sampled dX and dW entries, each from the lines
    of dY, W and X it contracts, quantized by the oracle along its own
    contraction axis."""
    import block_scaled_precision_gemm_gb300 as bsmm
    wl = bench.BackwardWork(W.BACKWARD, device)
    wl.step()
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    p = wl.p
    rng = _rng(3)
    fp8 = p.fp8

    def q_line(v, fmt):  # one contraction line (length multiple of 32), blocks of 32
        c, s = Q.quantize(v[None, :], (1, 32), fmt, "ue8m0")
        return G.scaled_operand(F.decode(c, fmt), F.decode(s, "ue8m0"))[0]

    ms, ks = rng.integers(0, p.M, N_SAMPLES), rng.integers(0, p.K, N_SAMPLES)
    got, ref, bnd = [], [], []
    for m, k in zip(ms, ks):
        dy = wl.dY[m].float().cpu().numpy()
        wcol = wl.W[:, k].float().cpu().numpy()
        prod = q_line(dy, fmt=fp8) * q_line(wcol, fmt=fp8)
        got.append(wl.dX[m, k].float().item()); ref.append(prod.sum()); bnd.append(np.abs(prod).sum())
    _check(np.array(got), np.array(ref), np.array(bnd), "dX", G.BF16_HALF_ULP)
    ns, ks = rng.integers(0, p.N, N_SAMPLES), rng.integers(0, p.K, N_SAMPLES)
    got, ref, bnd = [], [], []
    for n, k in zip(ns, ks):
        dycol = wl.dY[:, n].float().cpu().numpy()
        xcol = wl.X[:, k].float().cpu().numpy()
        prod = q_line(dycol, fmt=fp8) * q_line(xcol, fmt=fp8)
        got.append(wl.dW[n, k].float().item()); ref.append(prod.sum()); bnd.append(np.abs(prod).sum())
    _check(np.array(got), np.array(ref), np.array(bnd), "dW", G.BF16_HALF_ULP)
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
