"""The seeded input generators (workloads/), which both the CUDA path and the
oracle take their inputs from: deterministic, independent across roles, and
drawn with the shapes and distributions the input recipe states (the pages'
workloads: block_scaled_mm Input Generation and Shapes table; TensorTonic's
per-channel INT8 matmul; jax.nn.scaled_matmul's MXFP8/NVFP4 formats; the NKI
MXFP8 backward)."""
import math

import pytest
import torch

import workloads as W


def test_draws_are_deterministic_and_roles_independent():
    p = W.Grouped(64, 256, 256)
    a1, b1 = W.grouped_raw(p, 0)
    a2, b2 = W.grouped_raw(p, 0)
    assert torch.equal(a1, a2) and torch.equal(b1, b2)
    a3, _ = W.grouped_raw(p, 1)
    assert not torch.equal(a1, a3)                      # another seed
    assert not torch.equal(a1[:, :256], b1[:64, :256])  # another role
    a4, _ = W.grouped_raw(W.Grouped(64, 512, 256), 0)
    assert not torch.equal(a1, a4)                      # another problem of one workload


def test_grouped_draws_are_standard_normal_float32():
    a, b = W.grouped_raw(W.Grouped(4096, 256, 512), 2)
    assert a.dtype == b.dtype == torch.float32 and a.shape == (4096, 512) and b.shape == (256, 512)
    assert abs(a.mean().item()) < 0.01 and abs(a.std().item() - 1) < 0.01


def test_int8_zeroes_one_percent_of_x_rows_and_w_columns():
    p = W.Int8Channel(1000, 300, 500)
    x, w = W.int8_raw(p, 1)
    assert x.shape == (1000, 300) and w.shape == (300, 500) and x.dtype == w.dtype == torch.float32
    zero_rows = (x == 0).all(dim=1)
    zero_cols = (w == 0).all(dim=0)
    assert zero_rows.sum().item() == 10 and zero_cols.sum().item() == 5
    assert not (x[~zero_rows] == 0).any() and not (w[:, ~zero_cols] == 0).any()
    assert W.zero_lines(4096, 0.01, 1, W.S_ZERO_ROWS).numel() == 41
    assert W.zero_lines(20, 0.01, 1, W.S_ZERO_ROWS).numel() == 1  # at least one line


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_batched_draws(fmt):
    p = W.Batched(2, 64, 32, 512, fmt)
    a, b, sa, sb = W.batched_raw(p, 3)
    if fmt == "mxfp8":
        assert a.shape == (2, 64, 512) and a.dtype == torch.float32
    else:  # two E2M1 codes a byte, every byte value possible
        assert a.shape == (2, 64, 256) and a.dtype == torch.uint8
        assert a.min().item() == 0 and a.max().item() == 255
    if fmt == "nvfp4":  # scale values 2^u, u uniform in [-4, 4], one per 16-block
        assert sa.shape == (2, 64, 32) and sa.dtype == torch.float32
        u = torch.log2(torch.cat([sa.flatten(), sb.flatten()]))
        assert u.min().item() >= -4 and u.max().item() <= 4 and u.min().item() < -3.9 and u.max().item() > 3.9
    else:  # UE8M0 exponents uniform over -6..6, one per 32-block
        assert sa.shape == (2, 64, 16) and sa.dtype == torch.int32
        e = torch.cat([sa.flatten(), sb.flatten()])
        assert set(e.unique().tolist()) == set(range(-6, 7))
    assert b.shape[1] == 32


def test_backward_draws():
    dY, Wt, X = W.backward_raw(W.Backward(256, 384, 512), 4)
    assert dY.shape == (256, 384) and Wt.shape == (384, 512) and X.shape == (256, 512)
    assert dY.dtype == Wt.dtype == X.dtype == torch.bfloat16
    assert abs(dY.float().std().item() - 1) < 0.02
    assert abs(Wt.float().std().item() - 0.02) < 0.001 and abs(X.float().std().item() - 0.02) < 0.001


def test_workload_table_follows_the_pages_shapes():
    sweep = W.GROUPED_SWEEP.problems
    assert [(p.m, p.n, p.k) for p in sweep] == (
        [(m, 2048, 2048) for m in (349, 4533, 65536, 704512)] + [(m, 4096, 4096) for m in (237, 4096, 65536, 299520)])
    assert all(p.group_n == p.group_k == 128 for p in sweep)
    assert W.GROUPED_SMALL.problems == (W.Grouped(64, 256, 256),)
    assert W.INT8_4096.problems == (W.Int8Channel(4096, 4096, 4096),)
    assert W.MXFP8_BATCHED.problems == (W.Batched(8, 4096, 4096, 8192, "mxfp8"),)
    assert W.NVFP4_SQUARE.problems == (W.Batched(1, 16384, 16384, 16384, "nvfp4"),)
    assert W.BACKWARD.problems == (W.Backward(16384, 8192, 8192),)
    assert math.isclose(sum(2.0 * p.m * p.n * p.k for p in sweep) / 1e12, 18.9, rel_tol=0.01)
    assert len(W.WORKLOADS) == 7 and len({w.name for w in W.WORKLOADS.values()}) == 7
