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
