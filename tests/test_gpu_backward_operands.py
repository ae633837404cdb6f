"""The four operands bsmm_linear_backward quantizes into its workspace, read
back through the workspace layout include/bsmm.h documents, against the
oracle's quantizer bit for bit (NKI "Matmul MXFP8 Backward Kernel API
Reference", introduction: every operand MXFP8-quantized along its own GEMM's
contraction axis).

dY is quantized along both of its axes in one pass over it (the dual
quantizer): along N for dX = dY W, and along M, stored transposed, for
dW = dY^T X.  W and X are quantized along N and M, stored transposed.  Codes
must match the oracle's exactly; the UE8M0 scales, written straight into the
tensor-core atom layout, must decode to the oracle's scale bytes, with the
neutral scale in every padding byte.  The shapes include M and N that are not
multiples of the quantizer's 128 x 128 tiles."""

import numpy as np
import pytest
import torch

from oracle import gemm as G

from test_gpu_atoms import decode_atoms

pytestmark = pytest.mark.gpu


def _align(n, a=256):
    return (n + a - 1) // a * a


@pytest.mark.parametrize("fp8", ["e5m2", "e4m3"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (160, 96, 224), (512, 384, 256), (2048, 1056, 512)])
def test_backward_workspace_operands_match_oracle(fp8, M, N, K):
    import block_scaled_precision_gemm_gb300 as bsmm
    g = torch.Generator().manual_seed(M * 3 + N * 5 + K)
    dY = (torch.randn(M, N, generator=g) * 4).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    X = (torch.randn(M, K, generator=g) * 0.02).to(torch.bfloat16)
    ws = torch.full((bsmm.linear_backward_workspace_size(M, N, K),), 0xA5, dtype=torch.uint8, device="cuda")
    bsmm.linear_backward(dY.cuda(), W.cuda(), X.cuda(), fp8, workspace=ws)
    torch.cuda.synchronize()
    assert bsmm.check_device_status()[0] == 0
    buf = ws.cpu().numpy()
    dYf, Wf, Xf = dY.float().numpy(), W.float().numpy(), X.float().numpy()
    fmt = "mxfp8" if fp8 == "e4m3" else "mxfp8_e5m2"
    off = 0
    # the header's order: dY along N [M, N], W^T [K, N], dY^T [N, M], X^T [K, M],
    # each followed by its atoms, every part on a 256-byte boundary
    for name, src, axis, (rows, cols) in (("dY along N", dYf, "cols", (M, N)), ("W^T", Wf, "rows", (K, N)),
                                          ("dY^T", dYf, "rows", (N, M)), ("X^T", Xf, "rows", (K, M))):
        codes = buf[off:off + rows * cols].reshape(rows, cols)
        off += _align(rows * cols)
        n_atoms = bsmm.scale_atoms_size(1, rows, cols, fp8, "ue8m0")
        atoms = buf[off:off + n_atoms]
        off += _align(n_atoms)
        oc, osc = G.mx_quantize(src, axis, fp8)
        bad = np.argwhere(codes != oc)
        assert bad.size == 0, f"{name}: {len(bad)} codes differ, first at {bad[:4].tolist()}"
        np.testing.assert_array_equal(decode_atoms(atoms, 1, rows, cols, fmt)[0], osc, err_msg=f"{name} scales")
    assert off <= buf.size
