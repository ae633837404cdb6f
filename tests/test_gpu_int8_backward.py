"""GPU INT8 per-channel matmul and MXFP8 linear backward vs the oracle, and
the bounded-wait timeout path."""

import json
import os

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as G
from tests.conftest import GOLDEN

pytestmark = pytest.mark.gpu


def _bsmm():
    import block_scaled_precision_gemm_gb300 as bsmm
    return bsmm


def run_int8(x, w):
    bsmm = _bsmm()
    out = bsmm.int8_channel(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), return_acc=True)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    ref = G.int8_channel(x, w)
    np.testing.assert_array_equal(got["x_q"], ref["x_q"])
    np.testing.assert_array_equal(got["w_q"], ref["w_q"])
    np.testing.assert_array_equal(got["x_scales"].view(np.uint32), ref["x_scales"].view(np.uint32))
    np.testing.assert_array_equal(got["w_scales"].view(np.uint32), ref["w_scales"].view(np.uint32))
    np.testing.assert_array_equal(got["acc"].astype(np.int64), ref["acc"])
    # TensorTonic checker: relative 1e-6 of acc*sx*sw in float64; zero sum -> exactly 0
    y = got["y"].astype(np.float64)
    assert (np.abs(y - ref["y_ref"]) <= 1e-6 * np.abs(ref["y_ref"])).all()
    assert (got["y"][ref["acc"] == 0] == 0).all()
    return got


@pytest.mark.parametrize("i", [0, 1, 2])
def test_int8_worked_examples(i):
    with open(os.path.join(GOLDEN, "int8_per_channel_examples.json")) as f:
        ex = json.load(f)["examples"][i]
    got = run_int8(np.array(ex["x"], np.float32), np.array(ex["w"], np.float32))
    np.testing.assert_array_equal(got["x_q"], ex["x_q"])
    np.testing.assert_array_equal(got["w_q"], ex["w_q"])
    np.testing.assert_allclose(got["y"], ex["y"], rtol=0, atol=0.5e-6)


@pytest.mark.parametrize("B,D_in,D_out", [(100, 300, 70), (129, 256, 200), (6, 64, 6), (257, 1000, 130)])
def test_int8_random_with_zero_lines(B, D_in, D_out):
    g = torch.Generator().manual_seed(B + D_in)
    x = torch.randn(B, D_in, generator=g).numpy()
    w = torch.randn(D_in, D_out, generator=g).numpy()
    x[B // 2] = 0
    w[:, D_out // 3] = 0
    run_int8(x, w)


def test_int8_extreme_sums_stay_exact():
    """All codes +-127: |sum| = D_in * 16129 (the page's constraint scaled
    to D_in = 4096 is 66,064,384 < 2^31)."""
    x = np.ones((130, 4096), np.float32)
    w = np.ones((4096, 129), np.float32)
    w[:, 1::2] = -1
    got = run_int8(x, w)
    assert got["acc"][0, 0] == 4096 * 127 * 127 and got["acc"][0, 1] == -4096 * 127 * 127


@pytest.mark.parametrize("kernel", ["tc", "mma"])
@pytest.mark.parametrize("B,D_in,D_out", [(100, 300, 72), (6, 64, 8), (257, 1000, 132), (300, 4133, 264),
                                          (520, 2048, 516), (1, 128, 4),
                                          # D_out % 16 == 0: the fused column-strip quantizer
                                          (100, 300, 80), (257, 1000, 144), (300, 4133, 256), (1, 37, 16)])
def test_int8_each_kernel(monkeypatch, kernel, B, D_in, D_out):
    """The bf16 tensor-core path (exact FP32 chunks of 1024 products added in
    int32) and the mma.sync fallback, each forced, on ragged B / D_in / D_out
    with D_out % 4 == 0 (the tensor-core path's TMA stores)."""
    if kernel == "mma":
        monkeypatch.setenv("BSMM_INT8_KERNEL", "mma")
    g = torch.Generator().manual_seed(B * 7 + D_in)
    x = torch.randn(B, D_in, generator=g).numpy()
    w = torch.randn(D_in, D_out, generator=g).numpy()
    x[B // 3] = 0
    w[:, D_out // 2] = 0
    run_int8(x, w)


@pytest.mark.parametrize("B,D_in,D_out", [(64, 4096, 4096), (100, 300, 72), (7, 1000, 4100), (130, 3968, 36),
                                          (1, 64, 4), (33, 2048, 1028)])
def test_int8_w_quantizer_shapes(B, D_in, D_out):
    """w's per-column quantizer (rows held in registers for D_in <= 4096)
    over many strips (D_out 4096 and 4100), a partial last strip (D_out not
    a multiple of 32), column scales spread over e^[-4, 4] and a zero
    column."""
    g = torch.Generator().manual_seed(B + 3 * D_in + D_out)
    x = torch.randn(B, D_in, generator=g).numpy()
    w = (torch.randn(D_in, D_out, generator=g) * torch.exp(torch.empty(1, D_out).uniform_(-4, 4, generator=g))).numpy()
    w[:, D_out // 3] = 0
    run_int8(x, w)


@pytest.mark.parametrize("D_in", [4096, 4096 + 1000])
def test_int8_extreme_sums_tensor_core_path(D_in):
    """Codes all +-127 on the tensor-core path: every 1024-product chunk sums
    to +-16,516,096, within 2^24 of zero by 260,120, and the int32 totals
    reach +-D_in * 16129."""
    x = np.ones((260, D_in), np.float32)
    x[1::2] = -1
    w = np.ones((D_in, 132), np.float32)
    w[:, 1::2] = -1
    got = run_int8(x, w)
    assert got["acc"][0, 0] == D_in * 127 * 127 and got["acc"][1, 0] == -D_in * 127 * 127


@pytest.mark.parametrize("B,D_in,D_out", [(2304, 1100, 2304), (2400, 2100, 2080)])
def test_int8_more_tiles_than_clusters(B, D_in, D_out):
    """More 256 x 256 tiles (81, 90) than clusters (76 on GB300), a partial
    last wave, and K over two exact 16-block chunks: sums, codes and y stay
    exact."""
    g = np.random.default_rng(B + D_out)
    x = g.standard_normal((B, D_in)).astype(np.float32)
    w = g.standard_normal((D_in, D_out)).astype(np.float32)
    run_int8(x, w)


@pytest.mark.parametrize("B,D_in,D_out", [(1024, 4096, 1280), (2304, 4096, 2304), (1, 5000, 2048)])
def test_int8_split_tail_tiles_reused_workspace(B, D_in, D_out):
    """The tiles of the matmul's last, partial wave split K over the idle
    clusters (76 on GB300): 20 tiles in halves of 32 K blocks (two exact
    chunks each), 81 tiles with a tail of 5 in quarters of 16, 8 tiles of one
    row in parts of 32, 32 and 16 K blocks.  Every part leaves its int32 sums in the workspace and the last
    one of each warp slot adds them, so the workspace is handed over full of
    garbage and then reused for a second call on other inputs: sums, codes
    and y must be the oracle's both times."""
    bsmm = _bsmm()
    g = np.random.default_rng(B + D_in + D_out)
    ws = torch.full((bsmm.int8_channel_workspace_size(B, D_in, D_out),), 0xA5, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        x = g.standard_normal((B, D_in)).astype(np.float32)
        w = g.standard_normal((D_in, D_out)).astype(np.float32)
        x[B // 2] = 0
        out = bsmm.int8_channel(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), return_acc=True, workspace=ws)
        torch.cuda.synchronize()
        assert bsmm.check_device_status()[0] == 0
        ref = G.int8_channel(x, w)
        np.testing.assert_array_equal(out["acc"].cpu().numpy().astype(np.int64), ref["acc"])
        np.testing.assert_array_equal(out["x_q"].cpu().numpy(), ref["x_q"])
        np.testing.assert_array_equal(out["w_q"].cpu().numpy(), ref["w_q"])
        y = out["y"].cpu().numpy().astype(np.float64)
        assert (np.abs(y - ref["y_ref"]) <= 1e-6 * np.abs(ref["y_ref"])).all()


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def run_backward(dY, W, X, fp8="e5m2"):
    bsmm = _bsmm()
    tdY, tW, tX = _bf16(dY), _bf16(W), _bf16(X)
    dX, dW = bsmm.linear_backward(tdY.cuda(), tW.cuda(), tX.cuda(), fp8)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    ref = G.linear_backward(tdY.float().numpy(), tW.float().numpy(), tX.float().numpy(), fp8)
    return dX.float().cpu().numpy(), dW.float().cpu().numpy(), ref


def test_backward_exact_on_representable_inputs():
    rng = np.random.default_rng(12)
    M, N, K = 64, 96, 32
    dY = rng.integers(-2, 3, (M, N)).astype(np.float32)
    W = rng.integers(-2, 3, (N, K)).astype(np.float32)
    X = rng.integers(-2, 3, (M, K)).astype(np.float32)
    dX, dW, _ = run_backward(dY, W, X)
    np.testing.assert_array_equal(dX, dY @ W)
    np.testing.assert_array_equal(dW, dY.T @ X)


@pytest.mark.parametrize("M,N,K,fp8", [(128, 96, 160, "e5m2"), (256, 384, 128, "e5m2"), (96, 64, 320, "e4m3")])
def test_backward_parity(M, N, K, fp8):
    g = torch.Generator().manual_seed(M + N + K)
    dY = torch.randn(M, N, generator=g).numpy()
    W = (torch.randn(N, K, generator=g) * 0.02).numpy()
    X = (torch.randn(M, K, generator=g) * 0.02).numpy()
    dX, dW, ref = run_backward(dY, W, X, fp8)
    for got, y_ref, bound, name in ((dX, ref["dX"], ref["dX_bound"], "dX"), (dW, ref["dW"], ref["dW_bound"], "dW")):
        ok = G.within_bound(got, y_ref, bound, out_round=G.BF16_HALF_ULP)
        assert ok.all(), f"{name}: {(~ok).sum()} entries outside the bound"


def test_backward_quantized_operands_match_oracle():
    """The four MXFP8 operands the backward builds (quantizer with the same
    arguments) are bit-exact against the oracle's."""
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(77)
    M, N, K = 96, 64, 128
    dY = torch.randn(M, N, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    X = (torch.randn(M, K, generator=g) * 0.02).to(torch.bfloat16)
    ref = G.linear_backward(dY.float().numpy(), W.float().numpy(), X.float().numpy())
    c, s = bsmm.quantize(X.cuda(), (32, 1), "e5m2", "ue8m0", transpose=True)
    np.testing.assert_array_equal(c.cpu().numpy(), ref["xt"])
    np.testing.assert_array_equal(s.cpu().numpy(), ref["xt_s"])
    c, s = bsmm.quantize(dY.cuda(), (1, 32), "e5m2", "ue8m0")
    np.testing.assert_array_equal(c.cpu().numpy(), ref["dy_n"])
    np.testing.assert_array_equal(s.cpu().numpy(), ref["dy_n_s"])
    c, s = bsmm.quantize(W.cuda(), (32, 1), "e5m2", "ue8m0", transpose=True)
    np.testing.assert_array_equal(c.cpu().numpy(), ref["wt"])
    np.testing.assert_array_equal(s.cpu().numpy(), ref["wt_s"])
    c, s = bsmm.quantize(dY.cuda(), (32, 1), "e5m2", "ue8m0", transpose=True)
    np.testing.assert_array_equal(c.cpu().numpy(), ref["dyt"])
    np.testing.assert_array_equal(s.cpu().numpy(), ref["dyt_s"])


def test_bounded_wait_gives_up_and_context_survives():
    bsmm = _bsmm()
    assert bsmm.check_device_status()[0] == 0
    bsmm.selftest_wait_timeout(20_000_000)  # 20 ms, on a barrier nothing arrives on
    st, site = bsmm.check_device_status()
    assert st == bsmm.ERR_TIMEOUT and site == 7
    assert bsmm.check_device_status()[0] == 0          # cleared
    # the context is still usable
    a = torch.zeros((1, 32), dtype=torch.uint8, device="cuda")
    s = torch.full((1, 1), 127, dtype=torch.uint8, device="cuda")
    y = bsmm.gemm(a, a, s, s, "e4m3", "e4m3", "ue8m0")
    assert y.cpu().item() == 0.0


def test_int8_empty_batch_still_quantizes_w():
    """B == 0: no rows of x, y is empty, and w_q / w_scales are still the
    page's per-column codes and scales (bit-exact)."""
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(9)
    w = torch.randn((200, 24), generator=g).numpy()
    w[:, 5] = 0
    out = bsmm.int8_channel(torch.zeros((0, 200), device="cuda"), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert out["y"].shape == (0, 24) and bsmm.check_device_status()[0] == 0
    ref = G.int8_channel(np.zeros((1, 200), np.float32), w)
    np.testing.assert_array_equal(out["w_q"].cpu().numpy(), ref["w_q"])
    np.testing.assert_array_equal(out["w_scales"].cpu().numpy().view(np.uint32), ref["w_scales"].view(np.uint32))
