"""Per-kernel timing (bsmm_trace_*): every kernel a call launches shows up
once, by name, with a positive duration, including those on the INT8 call's
second stream; nothing is recorded once tracing is off."""

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_int8_call_records_its_kernels():
    import block_scaled_precision_gemm_gb300 as bsmm
    x = torch.randn(512, 1024, device="cuda")
    w = torch.randn(1024, 768, device="cuda")
    bsmm.int8_channel(x, w)  # set-up outside the trace
    with bsmm.trace() as launches:
        bsmm.int8_channel(x, w)
    names = [n for n, _, _ in launches]
    assert names.count("i8_quant_rows_reg") == 1
    assert names.count("i8_quant_w_strip") == 1
    assert names.count("tc_gemm_pair<I8>") == 1
    assert all(ms > 0 for _, _, ms in launches)
    assert launches[0][1] == 0.0 and all(t0 >= 0 for _, t0, _ in launches)
    bsmm.int8_channel(x, w)
    assert bsmm.lib().bsmm_trace_count() == len(launches)  # off: nothing added


def test_quantize_and_gemm_record_in_order():
    import block_scaled_precision_gemm_gb300 as bsmm
    a = torch.randn(300, 512, device="cuda")
    b = torch.randn(256, 512, device="cuda")
    with bsmm.trace() as launches:
        qa, sa = bsmm.quantize(a, (1, 128), "e4m3", "f32")
        qb, sb = bsmm.quantize(b, (128, 128), "e4m3", "f32")
        bsmm.gemm_grouped(qa, qb, sa, sb)
    names = [n for n, _, _ in launches]
    assert names[:2] == ["quant_rows", "quant_tile"]
    assert names[2].startswith("tc_gemm")
    starts = [t0 for _, t0, _ in launches]
    assert starts == sorted(starts)


def test_quantize_batch_shares_launches():
    """Three 128 x 128 jobs of one input type and scale kind run as one
    quant_tile_batch launch; a job of another kind gets its own, and a row
    quantization runs as bsmm_quantize runs it."""
    import block_scaled_precision_gemm_gb300 as bsmm
    jobs = [{"x": torch.randn(256, 384, device="cuda"), "block": (128, 128)} for _ in range(3)]
    jobs.append({"x": torch.randn(128, 256, device="cuda").bfloat16(), "block": (128, 128), "scale": "ue8m0"})
    jobs.append({"x": torch.randn(64, 256, device="cuda"), "block": (1, 128)})
    bsmm.quantize_batch(jobs)
    with bsmm.trace() as launches:
        bsmm.quantize_batch(jobs)
    names = sorted(n for n, _, _ in launches)
    assert names == ["quant_rows", "quant_tile_batch", "quant_tile_batch"]
