"""Calls from several host threads and inside CUDA graphs (include/bsmm.h:
calls are asynchronous on their stream and safe from several host threads;
the INT8 call forks part of its work onto a stream of the library and joins
it back, so it stays ordered on the caller's stream, graph capture
included)."""
import threading

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _bsmm():
    import block_scaled_precision_gemm_gb300 as bsmm
    return bsmm


def _int8_inputs(seed, B=512, D_in=1024, D_out=768):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, D_in, generator=g).cuda(), torch.randn(D_in, D_out, generator=g).cuda()


def test_int8_from_two_host_threads():
    bsmm = _bsmm()
    inputs = [_int8_inputs(s) for s in range(4)]
    ref = []
    for x, w in inputs:
        out = bsmm.int8_channel(x, w, return_acc=True)
        torch.cuda.synchronize()
        ref.append({k: v.clone() for k, v in out.items()})
    errors = []

    def worker(tid):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for it in range(10):
                    i = (tid + it) % len(inputs)
                    out = bsmm.int8_channel(*inputs[i], return_acc=True, stream=stream)
                    stream.synchronize()
                    for k, v in out.items():
                        if not torch.equal(v, ref[i][k]):
                            errors.append(f"thread {tid} call {it}: {k} differs")
        except Exception as e:  # reported below, not lost in the thread
            errors.append(f"thread {tid}: {e!r}")

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:5]
    assert bsmm.check_device_status()[0] == 0


def test_int8_in_a_cuda_graph():
    bsmm = _bsmm()
    x, w = _int8_inputs(7)
    out = bsmm.int8_channel(x, w, return_acc=True)  # eager, also creates the library's side stream
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in out.items()}
    ws = torch.empty(bsmm.int8_channel_workspace_size(*x.shape, w.shape[1]), dtype=torch.uint8, device="cuda")
    outs = {k: torch.empty_like(v) for k, v in out.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bsmm.int8_channel(x, w, return_acc=True, out=outs, workspace=ws)
    for v in outs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(outs[k], ref[k]), k


def test_mx_gemm_in_a_cuda_graph():
    bsmm = _bsmm()
    g = torch.Generator().manual_seed(3)
    xa = torch.randn(512, 1024, generator=g).cuda()
    xb = torch.randn(768, 1024, generator=g).cuda()
    ca, sa = bsmm.quantize(xa, (1, 32), "e4m3", "ue8m0")
    cb, sb = bsmm.quantize(xb, (1, 32), "e4m3", "ue8m0")
    y_ref = bsmm.gemm(ca, cb, sa, sb)
    torch.cuda.synchronize()
    y = torch.empty_like(y_ref)
    ws = torch.empty(bsmm.gemm_workspace_size(1, 512, 768, 1024, "e4m3"), dtype=torch.uint8, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bsmm.gemm(ca, cb, sa, sb, y=y, workspace=ws)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
    assert np.isfinite(y.cpu().numpy()).all()
