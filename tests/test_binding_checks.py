"""The binding's argument checks (include/bsmm.h takes raw pointers, so the
binding checks each tensor's shape, element type and size, then that all are
CUDA tensors on the current device, before any pointer reaches the library).

These run on CPU tensors: a malformed argument must be refused before any
device work, and a well-formed set must get as far as the device check."""
import pytest
import torch

import block_scaled_precision_gemm_gb300 as bsmm


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()  # incremental: the size queries below call into the library


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def refused(fn, *args, match, **kw):
    with pytest.raises((ValueError, TypeError), match=match):
        fn(*args, **kw)


CUDA = "must be a CUDA tensor"


def test_quantize_checks():
    refused(bsmm.quantize, f32(4, 64).to(torch.float64), (1, 32), match="float32 or")
    refused(bsmm.quantize, f32(4, 64), (1, 32), codes=u8(4, 63), match="codes must have shape")
    refused(bsmm.quantize, f32(4, 64), (1, 32), "e2m1", "ue4m3", codes=u8(4, 64), match="shape \\(4, 32\\)")
    refused(bsmm.quantize, f32(4, 64), (1, 32), "e4m3", "f32", scales=u8(4, 2), match="4-byte elements")
    refused(bsmm.quantize, f32(4, 64), (32, 1), transpose=True, scales=f32(4, 2), match="shape \\(64, 0\\)")
    refused(bsmm.quantize, f32(4, 64), (1, 32), match=CUDA)


def test_quantize_batch_checks():
    """Each job is checked, in order, as quantize() checks its arguments,
    before the call reaches the library; a missing required key is refused
    too."""
    good = {"x": f32(4, 64), "block": (1, 32)}
    refused(bsmm.quantize_batch, [{"x": f32(4, 64), "block": (1, 32), "codes": u8(4, 63)}, good],
            match="codes must have shape")
    refused(bsmm.quantize_batch, [{"x": f32(4, 64).to(torch.float64), "block": (1, 32)}], match="float32 or")
    with pytest.raises(KeyError):
        bsmm.quantize_batch([{"x": f32(4, 64)}])
    refused(bsmm.quantize_batch, [good], match=CUDA)


def test_gemm_checks():
    a, b, sa, sb = u8(2, 128, 256), u8(2, 64, 256), u8(2, 128, 8), u8(2, 64, 8)
    refused(bsmm.gemm, a, u8(2, 64, 255), sa, sb, match="b must have shape \\(2, 64, 256\\)")
    refused(bsmm.gemm, a, u8(1, 64, 256), sa, sb, match="b must have shape")
    refused(bsmm.gemm, a, b, u8(2, 127, 8), sb, match="a_scales must have shape")
    refused(bsmm.gemm, a, b, sa, f32(2, 64, 8), match="1-byte elements")
    refused(bsmm.gemm, a, b, sa, sb, y=f32(2, 128, 63), match="y must have shape")
    refused(bsmm.gemm, a, b, sa, sb, y=torch.zeros(2, 128, 64, dtype=torch.float16), match="y must be")
    refused(bsmm.gemm, a.float(), b, sa, sb, match="1-byte elements")
    refused(bsmm.gemm, a, b, sa, sb, K=512, match="a must have shape")
    # E2M1 packs two codes a byte: K = 2 x the last dimension
    refused(bsmm.gemm, u8(1, 128, 128), u8(1, 64, 256), u8(1, 128, 16), u8(1, 64, 16), "e2m1", "e2m1", "ue4m3",
            match="b must have shape \\(1, 64, 128\\)")
    refused(bsmm.gemm, a, b, sa, sb, match=CUDA)
    refused(bsmm.gemm, a[0], b[0], sa[0], sb[0], match=CUDA)  # 2-D operands: one batch
    refused(bsmm.gemm_noalloc, a, b, sa, sb, match="needs y")
    refused(bsmm.gemm_noalloc, a, b, sa, sb, y=f32(2, 128, 64), match=CUDA)


def test_gemm_grouped_checks():
    a, b = u8(256, 512), u8(384, 512)
    sa, sb = f32(256, 4), f32(3, 4)
    refused(bsmm.gemm_grouped, a, u8(384, 256), sa, sb, match="b must have shape")
    refused(bsmm.gemm_grouped, a, b, f32(256, 3), sb, match="a_scales must have shape \\(256, 4\\)")
    refused(bsmm.gemm_grouped, a, b, sa, f32(4, 4), match="b_scales must have shape \\(3, 4\\)")
    refused(bsmm.gemm_grouped, a, b, sa, sb.to(torch.bfloat16), match="b_scales must be")
    refused(bsmm.gemm_grouped, a, b, sa, sb, y=f32(256, 383), match="y must have shape")
    refused(bsmm.gemm_grouped, a, b, sa, sb, match=CUDA)


def test_int8_channel_checks():
    x, w = f32(16, 64), f32(64, 32)
    refused(bsmm.int8_channel, x, f32(63, 32), match="w must have shape \\(64, 32\\)")
    refused(bsmm.int8_channel, x.bfloat16(), w, match="x must be")
    refused(bsmm.int8_channel, x, w, out={"y": f32(16, 31)}, match="y.*must have shape")
    refused(bsmm.int8_channel, x, w, out={"x_q": u8(16, 64)}, match="x_q.*must be")
    refused(bsmm.int8_channel, x, w, out={"z": f32(1)}, match="unknown key")
    refused(bsmm.int8_channel, x, w, match=CUDA)


def test_linear_backward_checks():
    dY, W, X = bf16(64, 96), bf16(96, 128), bf16(64, 128)
    refused(bsmm.linear_backward, dY, bf16(95, 128), X, match="W must have shape")
    refused(bsmm.linear_backward, dY, W, bf16(64, 127), match="X must have shape")
    refused(bsmm.linear_backward, dY.float(), W, X, match="dY must be")
    refused(bsmm.linear_backward, dY, W, X, dX=bf16(64, 96), match="dX must have shape")
    refused(bsmm.linear_backward, dY, W, X, match=CUDA)


def test_quantize_atoms_checks():
    refused(bsmm.quantize_atoms, f32(300, 64), batches=7, match="do not split")
    refused(bsmm.quantize_atoms, f32(300, 64), batches=0, match="positive")
    refused(bsmm.quantize_atoms, f32(300, 64), codes=u8(300, 32), match="codes must have shape")
    refused(bsmm.quantize_atoms, f32(300, 64), match=CUDA)


def test_atom_entry_points_check_sizes(built):
    a, b = u8(1, 300, 384), u8(1, 200, 384)
    need_a = bsmm.scale_atoms_size(1, 300, 384)
    need_b = bsmm.scale_atoms_size(1, 200, 384)
    refused(bsmm.gemm_atoms, a, b, u8(need_a - 1), u8(need_b), match="a_atoms holds")
    refused(bsmm.gemm_atoms, a, b, u8(need_a), u8(need_b - 512), match="b_atoms holds")
    refused(bsmm.gemm_atoms, a, b, u8(need_a), u8(need_b), match=CUDA)
    M, N, K = 64, 96, 128
    q = dict(dy_n=u8(M, N), dy_n_scales=u8(M, N // 32), w_t=u8(K, N), w_t_scales=u8(K, N // 32),
             dy_t=u8(N, M), dy_t_scales=u8(N, M // 32), x_t=u8(K, M), x_t_scales=u8(K, M // 32))
    refused(bsmm.linear_backward_quantized, **{**q, "dy_t": u8(N, M + 1)}, match="dy_t must have shape")
    refused(bsmm.linear_backward_quantized, **{**q, "x_t_scales": u8(K, 3)}, match="x_t_scales must have shape")
    refused(bsmm.linear_backward_quantized, **q, match=CUDA)
    atoms = {k: (u8(bsmm.scale_atoms_size(1, *v.shape, "e5m2")) if not k.endswith("scales") else None)
             for k, v in q.items() if not k.endswith("scales")}
    qa = dict(q)
    for k in ("dy_n", "w_t", "dy_t", "x_t"):
        qa[k + "_scales"] = atoms[k]
    refused(bsmm.linear_backward_quantized, **{**qa, "w_t_scales": u8(1)}, scales_are_atoms=True,
            match="w_t_scales holds")
    refused(bsmm.linear_backward_quantized, **qa, scales_are_atoms=True, match=CUDA)
