"""Python binding of libbsmm.so, the block-scaled low-precision GEMM library.

Argument marshalling only: every function here checks what the library
cannot see through raw pointers (each tensor's shape, element type and size,
and that all are contiguous CUDA tensors on the current device), allocates
its outputs with torch (device memory is the caller's, as the C ABI
requires), passes raw device pointers and the current torch stream to the C
entry point of the same name, and raises :class:`BsmmError` on a non-zero
status.  Everything else (divisibility, formats, alignment, workspace size)
is the library's to check.  All computation happens in the
library's CUDA kernels; there is no CPU path.  The library is loaded on first
use and its absence is an error.

Entry points (see ``include/bsmm.h`` for the full contract):

* :func:`quantize`        absmax block quantizer (E4M3/E5M2/E2M1/INT8 codes,
                          FP32/UE8M0/UE4M3 scales, optional transposed output)
* :func:`gemm`            batched block-scaled GEMM, MXFP8 or NVFP4
* :func:`gemm_grouped`    FP8 GEMM with 1x128 / 128x128 FP32 scales
* :func:`int8_channel`    INT8 per-channel matmul with exact INT32 sums
* :func:`linear_backward` MXFP8 dX / dW of a linear layer
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "BsmmError", "lib", "library_path", "quantize", "quantize_batch", "gemm", "gemm_noalloc", "gemm_grouped", "int8_channel",
    "linear_backward", "gemm_workspace_size", "int8_channel_workspace_size",
    "linear_backward_workspace_size", "check_device_status", "selftest_wait_timeout", "selftest_quotient", "trace",
    "scale_atoms_size", "quantize_atoms", "gemm_atoms", "linear_backward_quantized",
    "set_wait_timeout_ns", "version",
    "F32", "BF16", "E4M3", "E5M2", "E2M1", "INT8", "SCALE_F32", "SCALE_UE8M0", "SCALE_UE4M3",
]

# bsmm_status
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(8)
STATUS_NAMES = ["OK", "INVALID_ARG", "SHAPE", "ALIGNMENT", "UNSUPPORTED", "CUDA", "TIMEOUT", "WORKSPACE"]
# bsmm_dtype
F32, BF16, E4M3, E5M2, E2M1, INT8 = range(6)
# bsmm_scale_type
SCALE_F32, SCALE_UE8M0, SCALE_UE4M3 = range(3)

_CODE_NAMES = {"e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1, "int8": INT8}
_SCALE_NAMES = {"f32": SCALE_F32, "ue8m0": SCALE_UE8M0, "ue4m3": SCALE_UE4M3}

library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libbsmm.so")
_LIB = None


class BsmmError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{where}: BSMM_ERR_{name}: {msg}")


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_SZ = ctypes.c_size_t


class _QuantizeJob(ctypes.Structure):
    """bsmm_quantize_job (include/bsmm.h)."""
    _fields_ = [("x", _P), ("x_type", _INT), ("rows", _I64), ("cols", _I64), ("ld_x", _I64),
                ("block_rows", _INT), ("block_cols", _INT), ("code_type", _INT), ("scale_type", _INT),
                ("transpose_out", _INT), ("codes", _P), ("ld_codes", _I64), ("scales", _P), ("ld_scales", _I64)]


_SIGS = {
    "bsmm_version": ([], _INT),
    "bsmm_last_error": ([], ctypes.c_char_p),
    "bsmm_set_wait_timeout_ns": ([ctypes.c_uint64], None),
    "bsmm_check_device_status": ([_P, ctypes.POINTER(_INT)], _INT),
    "bsmm_selftest_wait_timeout": ([ctypes.c_uint64, _P], _INT),
    "bsmm_selftest_quotient": ([ctypes.c_uint64, ctypes.c_uint64, _P, _P], _INT),
    "bsmm_trace_start": ([], _INT),
    "bsmm_trace_stop": ([], _INT),
    "bsmm_trace_count": ([], _INT),
    "bsmm_trace_read": ([_INT, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float),
                         ctypes.POINTER(ctypes.c_float)], _INT),
    "bsmm_quantize": ([_P, _INT, _I64, _I64, _I64, _INT, _INT, _INT, _INT, _INT, _P, _I64, _P, _I64, _P], _INT),
    "bsmm_quantize_batch": ([ctypes.POINTER(_QuantizeJob), _INT, _P], _INT),
    "bsmm_gemm_workspace_size": ([_I64, _I64, _I64, _I64, _INT], _SZ),
    "bsmm_gemm": ([_I64, _I64, _I64, _I64, _P, _INT, _P, _INT, _P, _I64, _P, _I64, _INT, _P, _INT, _P, _SZ, _P],
                  _INT),
    "bsmm_gemm_noalloc": ([_I64, _I64, _I64, _I64, _P, _INT, _P, _INT, _P, _I64, _P, _I64, _INT, _P, _INT, _P],
                          _INT),
    "bsmm_gemm_grouped": ([_I64, _I64, _I64, _P, _INT, _P, _INT, _P, _P, _INT, _INT, _P, _P], _INT),
    "bsmm_int8_channel_workspace_size": ([_I64, _I64, _I64], _SZ),
    "bsmm_int8_channel": ([_P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _INT),
    "bsmm_linear_backward_workspace_size": ([_I64, _I64, _I64], _SZ),
    "bsmm_linear_backward": ([_P, _P, _P, _I64, _I64, _I64, _INT, _P, _P, _P, _SZ, _P], _INT),
    "bsmm_scale_atoms_size": ([_I64, _I64, _I64, _INT, _INT], _SZ),
    "bsmm_quantize_atoms": ([_P, _INT, _I64, _I64, _I64, _INT, _INT, _INT, _P, _P, _SZ, _P], _INT),
    "bsmm_gemm_atoms": ([_I64, _I64, _I64, _I64, _P, _INT, _P, _INT, _P, _P, _INT, _P, _INT, _P, _SZ, _P], _INT),
    "bsmm_linear_backward_quantized_workspace_size": ([_I64, _I64, _I64, _INT], _SZ),
    "bsmm_linear_backward_quantized": ([_I64, _I64, _I64, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _INT, _P, _P, _P,
                                        _SZ, _P], _INT),
}


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        h = ctypes.CDLL(library_path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(h, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = h
    return _LIB


def _check(status: int, where: str) -> None:
    if status != OK:
        raise BsmmError(status, where, lib().bsmm_last_error().decode())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_FLOATS = (torch.float32, torch.bfloat16)


def _want(t, name: str, shape=None, dtypes=None, itemsize=None, min_bytes=None) -> torch.Tensor:
    """Checks a tensor argument's shape, dtype and size before its pointer is
    passed on: the library sees raw pointers only, so a buffer that is too
    small, or of another element type, would be read or written out of
    bounds on the device."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} must be {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if itemsize is not None and t.element_size() != itemsize:
        raise ValueError(f"{name} must have {itemsize}-byte elements, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(int(s) for s in shape):
        raise ValueError(f"{name} must have shape {tuple(int(s) for s in shape)}, got {tuple(t.shape)}")
    if min_bytes is not None and t.numel() * t.element_size() < min_bytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, {min_bytes} needed")
    return t


def _on_device(**named) -> torch.device:
    """All tensor arguments are contiguous CUDA tensors on the current device
    (the library launches on the current device); returns that device."""
    dev = None
    for name, t in named.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other arguments on {dev}")
    if dev is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"the arguments are on {dev}, the current device is cuda:{torch.cuda.current_device()}")
    return dev


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _code(c) -> int:
    return _CODE_NAMES[c] if isinstance(c, str) else int(c)


def _scale(s) -> int:
    return _SCALE_NAMES[s] if isinstance(s, str) else int(s)


def version() -> int:
    return lib().bsmm_version()


def set_wait_timeout_ns(ns: int) -> None:
    lib().bsmm_set_wait_timeout_ns(int(ns))


def check_device_status(stream=None):
    """Synchronizes the stream; returns (status, site) of the device status word."""
    where = ctypes.c_int(0)
    st = lib().bsmm_check_device_status(_stream(stream), ctypes.byref(where))
    return st, where.value


def selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(lib().bsmm_selftest_wait_timeout(int(timeout_ns), _stream(stream)), "bsmm_selftest_wait_timeout")


# --------------------------------------------------------------------------- #
# quantize                                                                    #
# --------------------------------------------------------------------------- #

def selftest_quotient(pairs: int, seed: int = 0, device=None) -> int:
    """Pairs on which the quantizers' block quotient disagrees with the
    hardware division (bsmm_selftest_quotient); 0 is the expected answer."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    bad = torch.zeros(1, dtype=torch.int64, device=dev)
    with torch.cuda.device(dev):
        _check(lib().bsmm_selftest_quotient(int(pairs), int(seed) & (2**64 - 1), _ptr(bad), _stream(None)),
               "bsmm_selftest_quotient")
        return int(bad.item())


class trace:
    """Per-kernel timing of everything the library launches inside the block
    (bsmm_trace_*): ``with trace() as launches: ...`` leaves in ``launches``
    one ``(kernel, start_ms, ms)`` per launch, in launch order, start
    relative to the first launch.  Reading them waits for those kernels."""

    def __enter__(self):
        self.launches = []
        _check(lib().bsmm_trace_start(), "bsmm_trace_start")
        return self.launches

    def __exit__(self, exc_type, exc, tb):
        L = lib()
        L.bsmm_trace_stop()
        if exc_type is not None:  # leave the records unread; the block's exception propagates
            return False
        for i in range(L.bsmm_trace_count()):
            name, t0, ms = ctypes.c_char_p(), ctypes.c_float(), ctypes.c_float()
            _check(L.bsmm_trace_read(i, ctypes.byref(name), ctypes.byref(t0), ctypes.byref(ms)), "bsmm_trace_read")
            self.launches.append((name.value.decode(), t0.value, ms.value))
        return False


def _quantize_job(x, block, code, scale, transpose, codes, scales):
    """Checked arguments of one quantization, its outputs (allocated where
    not given) and the C job that describes it."""
    _want(x, "x", dtypes=_FLOATS)
    if x.dim() != 2:
        raise ValueError("x must be a 2-D float32 or bfloat16 tensor")
    br, bc = int(block[0]), int(block[1])
    c, s = _code(code), _scale(scale)
    rows, cols = x.shape
    orows, ocols = (cols, rows) if transpose else (rows, cols)
    srows, scols = ((cols // bc, rows // br) if transpose else (rows // br, cols // bc)) if br > 0 and bc > 0 else (0, 0)
    width = ocols // 2 if c == E2M1 else ocols
    scale_dtype = torch.float32 if s == SCALE_F32 else torch.uint8
    if codes is not None:
        _want(codes, "codes", (orows, width), itemsize=1)
    if scales is not None:
        _want(scales, "scales", (srows, scols), itemsize=scale_dtype.itemsize)
    dev = _on_device(x=x, codes=codes, scales=scales)
    if codes is None:
        codes = torch.empty((orows, width), dtype=torch.int8 if c == INT8 else torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((srows, scols), dtype=scale_dtype, device=dev)
    job = _QuantizeJob(_ptr(x), BF16 if x.dtype == torch.bfloat16 else F32, rows, cols, cols, br, bc, c, s,
                       1 if transpose else 0, _ptr(codes), ocols, _ptr(scales), scols)
    return job, codes, scales


def quantize(x: torch.Tensor, block, code="e4m3", scale="f32", transpose=False, codes=None, scales=None,
             stream=None):
    """Block-quantize a 2-D float32/bfloat16 CUDA tensor.

    Returns ``(codes, scales)``: codes uint8 (int8 for INT8; E2M1 packed two
    per byte) of shape [rows, cols] (or [cols, rows] transposed), scales
    float32 or uint8 of shape [rows/br, cols/bc] (or transposed)."""
    j, codes, scales = _quantize_job(x, block, code, scale, transpose, codes, scales)
    _check(lib().bsmm_quantize(j.x, j.x_type, j.rows, j.cols, j.ld_x, j.block_rows, j.block_cols, j.code_type,
                               j.scale_type, j.transpose_out, j.codes, j.ld_codes, j.scales, j.ld_scales,
                               _stream(stream)), "bsmm_quantize")
    return codes, scales


def quantize_batch(jobs, stream=None):
    """Several independent quantizations in one call (bsmm_quantize_batch).

    ``jobs`` is a list of dicts with the arguments of :func:`quantize`
    (``x`` and ``block`` required; ``code``, ``scale``, ``transpose``,
    ``codes``, ``scales`` optional).  Returns the ``(codes, scales)`` pairs in
    job order."""
    prepared = [_quantize_job(j["x"], j["block"], j.get("code", "e4m3"), j.get("scale", "f32"),
                              j.get("transpose", False), j.get("codes"), j.get("scales")) for j in jobs]
    arr = (_QuantizeJob * max(len(prepared), 1))(*[p[0] for p in prepared])
    _check(lib().bsmm_quantize_batch(arr, len(prepared), _stream(stream)), "bsmm_quantize_batch")
    return [(p[1], p[2]) for p in prepared]


# --------------------------------------------------------------------------- #
# GEMMs                                                                       #
# --------------------------------------------------------------------------- #

def gemm_workspace_size(B, M, N, K, a_type) -> int:
    return lib().bsmm_gemm_workspace_size(B, M, N, K, _code(a_type))


def gemm(a, b, a_scales, b_scales, a_type="e4m3", b_type="e4m3", scale="ue8m0", out_dtype=torch.float32, y=None,
         workspace=None, K=None, stream=None):
    """Batched block-scaled GEMM ``(B,M,K) x (B,N,K) -> (B,M,N)``.

    ``a``/``b`` hold codes (uint8 or float8 tensors; E2M1 packed, so their last
    dimension is K/2 and ``K`` is inferred as twice it), ``a_scales``
    (B,M,K_a) / ``b_scales`` (B,N,K_b) hold scale bytes."""
    at, bt = _code(a_type), _code(b_type)
    a, b, a_scales, b_scales, Bn, M, N, K = _gemm_operands(a, b, a_scales, b_scales, at, bt, K)
    if y is not None:
        _want(y, "y", (Bn, M, N), dtypes=_FLOATS)
    if workspace is not None:
        _want(workspace, "workspace")
    dev = _on_device(a=a, b=b, a_scales=a_scales, b_scales=b_scales, y=y, workspace=workspace)
    if y is None:
        y = torch.empty((Bn, M, N), dtype=out_dtype, device=dev)
    if workspace is None:
        workspace = torch.empty(max(gemm_workspace_size(Bn, M, N, K, at), 1), dtype=torch.uint8, device=dev)
    _check(lib().bsmm_gemm(Bn, M, N, K, _ptr(a), at, _ptr(b), bt, _ptr(a_scales), a_scales.shape[-1],
                           _ptr(b_scales), b_scales.shape[-1], _scale(scale), _ptr(y),
                           BF16 if y.dtype == torch.bfloat16 else F32, _ptr(workspace), _nbytes(workspace),
                           _stream(stream)), "bsmm_gemm")
    return y


def _code_bytes(t: int, K: int) -> int:
    """Bytes of K codes of type t in a row (E2M1 packs two per byte)."""
    return K // 2 if t == E2M1 else K


def _gemm_operands(a, b, a_scales, b_scales, at, bt, K):
    """Batched GEMM operands: codes (B,M,K) and (B,N,K) bytes (E2M1: K/2),
    scales (B,M,K_a) and (B,N,K_b) bytes; 2-D operands are one batch."""
    for t, n in ((a, "a"), (b, "b")):
        _want(t, n, itemsize=1)
    if a.dim() == 2 and b.dim() == 2:
        a, b = a[None], b[None]
        a_scales = a_scales[None] if a_scales is not None and a_scales.dim() == 2 else a_scales
        b_scales = b_scales[None] if b_scales is not None and b_scales.dim() == 2 else b_scales
    if a.dim() != 3 or b.dim() != 3:
        raise ValueError("a and b must be (B, M, K) and (B, N, K) code tensors")
    Bn, M, ka = a.shape
    N = b.shape[1]
    if K is None:
        K = ka * 2 if at == E2M1 else ka
    _want(a, "a", (Bn, M, _code_bytes(at, K)))
    _want(b, "b", (Bn, N, _code_bytes(bt, K)))
    if a_scales is not None:  # row-major scales (the atom entry points pass None)
        for t, n, rows in ((a_scales, "a_scales", M), (b_scales, "b_scales", N)):
            _want(t, n, itemsize=1)
            if t.dim() != 3:
                raise ValueError(f"{n} must be (B, rows, K / block)")
            _want(t, n, (Bn, rows, t.shape[-1]))
    return a, b, a_scales, b_scales, Bn, M, N, K


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def gemm_noalloc(a, b, a_scales, b_scales, a_type="e4m3", b_type="e4m3", scale="ue8m0", y=None, K=None,
                 stream=None):
    """:func:`gemm` through the entry point that allocates nothing: its
    scratch is a static device array of NOALLOC_SCRATCH_BYTES inside the
    library (for callers that cannot allocate device memory).  ``y`` must be
    given; this wrapper allocates nothing either."""
    at, bt = _code(a_type), _code(b_type)
    a, b, a_scales, b_scales, Bn, M, N, K = _gemm_operands(a, b, a_scales, b_scales, at, bt, K)
    if y is None:
        raise ValueError("gemm_noalloc needs y")
    _want(y, "y", (Bn, M, N), dtypes=_FLOATS)
    _on_device(a=a, b=b, a_scales=a_scales, b_scales=b_scales, y=y)
    _check(lib().bsmm_gemm_noalloc(Bn, M, N, K, _ptr(a), at, _ptr(b), bt, _ptr(a_scales), a_scales.shape[-1],
                                   _ptr(b_scales), b_scales.shape[-1], _scale(scale), _ptr(y),
                                   BF16 if y.dtype == torch.bfloat16 else F32, _stream(stream)),
           "bsmm_gemm_noalloc")
    return y


def gemm_grouped(a, b, a_scales, b_scales, group_n=128, group_k=128, a_type="e4m3", b_type="e4m3", y=None,
                 stream=None):
    """``y[m,n] = sum_kb a_scales[m,kb] * b_scales[n//group_n,kb] * (a.b over block kb)``."""
    for t, n in ((a, "a"), (b, "b")):
        _want(t, n, itemsize=1)
        if t.dim() != 2:
            raise ValueError(f"{n} must be a 2-D code tensor")
    M, K = a.shape
    N = b.shape[0]
    _want(b, "b", (N, K))
    for t, n in ((a_scales, "a_scales"), (b_scales, "b_scales")):
        _want(t, n, dtypes=(torch.float32,))
    # an empty output reads no scales; indivisible groups: the library says why
    if M and N and group_n > 0 and group_k > 0 and N % group_n == 0 and K % group_k == 0:
        _want(a_scales, "a_scales", (M, K // group_k))
        _want(b_scales, "b_scales", (N // group_n, K // group_k))
    if y is not None:
        _want(y, "y", (M, N), dtypes=(torch.float32,))
    dev = _on_device(a=a, b=b, a_scales=a_scales, b_scales=b_scales, y=y)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _check(lib().bsmm_gemm_grouped(M, N, K, _ptr(a), _code(a_type), _ptr(b), _code(b_type), _ptr(a_scales),
                                   _ptr(b_scales), group_n, group_k, _ptr(y), _stream(stream)),
           "bsmm_gemm_grouped")
    return y


def int8_channel_workspace_size(B, D_in, D_out) -> int:
    return lib().bsmm_int8_channel_workspace_size(B, D_in, D_out)


def int8_channel(x, w, return_acc=False, out=None, workspace=None, stream=None) -> dict:
    """INT8 per-channel matmul; returns the dict of the page (w_q, w_scales,
    x_q, x_scales, y) plus ``acc`` (int32 sums) when ``return_acc``."""
    for t, n in ((x, "x"), (w, "w")):
        _want(t, n, dtypes=(torch.float32,))
        if t.dim() != 2:
            raise ValueError(f"{n} must be a 2-D float32 tensor")
    Bn, D_in = x.shape
    D_out = w.shape[1]
    _want(w, "w", (D_in, D_out))
    want = {"x_q": ((Bn, D_in), (torch.int8,)), "x_scales": ((Bn,), (torch.float32,)),
            "w_q": ((D_in, D_out), (torch.int8,)), "w_scales": ((D_out,), (torch.float32,)),
            "y": ((Bn, D_out), (torch.float32,)), "acc": ((Bn, D_out), (torch.int32,))}
    o = dict(out) if out else {}
    for k, t in o.items():
        if k not in want:
            raise ValueError(f"out has an unknown key {k!r}")
        _want(t, f"out[{k!r}]", *want[k])
    if workspace is not None:
        _want(workspace, "workspace")
    dev = _on_device(x=x, w=w, workspace=workspace, **{f"out_{k}": t for k, t in o.items()})
    for k in ("x_q", "x_scales", "w_q", "w_scales", "y") + (("acc",) if return_acc else ()):
        if k not in o:
            o[k] = torch.empty(want[k][0], dtype=want[k][1][0], device=dev)
    if workspace is None:
        workspace = torch.empty(max(int8_channel_workspace_size(Bn, D_in, D_out), 1), dtype=torch.uint8,
                                device=dev)
    _check(lib().bsmm_int8_channel(_ptr(x), _ptr(w), Bn, D_in, D_out, _ptr(o["x_q"]), _ptr(o["x_scales"]),
                                   _ptr(o["w_q"]), _ptr(o["w_scales"]), _ptr(o["y"]), _ptr(o.get("acc")),
                                   _ptr(workspace), _nbytes(workspace), _stream(stream)), "bsmm_int8_channel")
    if out is not None:  # the caller's dict gets the outputs allocated here too
        out.update(o)
        return out
    return o


def linear_backward_workspace_size(M, N, K) -> int:
    return lib().bsmm_linear_backward_workspace_size(M, N, K)


def linear_backward(dY, W, X, fp8="e5m2", dX=None, dW=None, workspace=None, stream=None):
    """MXFP8 backward of ``Y = X @ W^T``: returns ``(dX, dW)`` in bfloat16."""
    bf16 = (torch.bfloat16,)
    for t, n in ((dY, "dY"), (W, "W"), (X, "X")):
        _want(t, n, dtypes=bf16)
        if t.dim() != 2:
            raise ValueError(f"{n} must be a 2-D bfloat16 tensor")
    M, N = dY.shape
    K = W.shape[1]
    _want(W, "W", (N, K))
    _want(X, "X", (M, K))
    if dX is not None:
        _want(dX, "dX", (M, K), dtypes=bf16)
    if dW is not None:
        _want(dW, "dW", (N, K), dtypes=bf16)
    if workspace is not None:
        _want(workspace, "workspace")
    dev = _on_device(dY=dY, W=W, X=X, dX=dX, dW=dW, workspace=workspace)
    if dX is None:
        dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if dW is None:
        dW = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = torch.empty(max(linear_backward_workspace_size(M, N, K), 1), dtype=torch.uint8, device=dev)
    _check(lib().bsmm_linear_backward(_ptr(dY), _ptr(W), _ptr(X), M, N, K, _code(fp8), _ptr(dX), _ptr(dW),
                                      _ptr(workspace), _nbytes(workspace), _stream(stream)), "bsmm_linear_backward")
    return dX, dW


# --------------------------------------------------------------------------- #
# Scales in the tensor cores' atom layout                                     #
# --------------------------------------------------------------------------- #

def scale_atoms_size(B, rows, K, code="e4m3", scale="ue8m0") -> int:
    return lib().bsmm_scale_atoms_size(B, rows, K, _code(code), _scale(scale))


def quantize_atoms(x, code="e4m3", scale="ue8m0", batches=1, transpose=False, codes=None, atoms=None, stream=None):
    """Quantize a GEMM operand with its scales written in the atom layout.

    ``x`` is [batches * rows, K] (or [K, rows] with ``transpose``); returns
    ``(codes, atoms)``: codes [batches * rows, K] (E2M1 packed: K/2 bytes a
    row) and the atoms as a flat uint8 tensor."""
    _want(x, "x", dtypes=_FLOATS)
    if x.dim() != 2:
        raise ValueError("x must be a 2-D float32 or bfloat16 tensor")
    c, s = _code(code), _scale(scale)
    batches = int(batches)
    if batches < 1:
        raise ValueError("batches must be positive")
    if transpose:
        K, rows = x.shape
    else:
        total, K = x.shape
        if total % batches:
            raise ValueError(f"x's {total} rows do not split into {batches} batches")
        rows = total // batches
    if codes is not None:
        _want(codes, "codes", (batches * rows, _code_bytes(c, K)), itemsize=1)
    if atoms is not None:
        _want(atoms, "atoms")
    dev = _on_device(x=x, codes=codes, atoms=atoms)
    if codes is None:
        codes = torch.empty((batches * rows, _code_bytes(c, K)), dtype=torch.uint8, device=dev)
    if atoms is None:
        atoms = torch.empty(max(scale_atoms_size(batches, rows, K, c, s), 1), dtype=torch.uint8, device=dev)
    _check(lib().bsmm_quantize_atoms(_ptr(x), BF16 if x.dtype == torch.bfloat16 else F32, batches, rows, K,
                                     1 if transpose else 0, c, s, _ptr(codes), _ptr(atoms), _nbytes(atoms),
                                     _stream(stream)), "bsmm_quantize_atoms")
    return codes, atoms


def gemm_atoms(a, b, a_atoms, b_atoms, a_type="e4m3", b_type="e4m3", scale="ue8m0", out_dtype=torch.float32,
               y=None, workspace=None, K=None, stream=None):
    """:func:`gemm` with both operands' scales in the atom layout."""
    at, bt, sc = _code(a_type), _code(b_type), _scale(scale)
    a, b, _, _, Bn, M, N, K = _gemm_operands(a, b, None, None, at, bt, K)
    _want(a_atoms, "a_atoms", min_bytes=scale_atoms_size(Bn, M, K, at, sc))
    _want(b_atoms, "b_atoms", min_bytes=scale_atoms_size(Bn, N, K, bt, sc))
    if y is not None:
        _want(y, "y", (Bn, M, N), dtypes=_FLOATS)
    if workspace is not None:
        _want(workspace, "workspace")
    dev = _on_device(a=a, b=b, a_atoms=a_atoms, b_atoms=b_atoms, y=y, workspace=workspace)
    if y is None:
        y = torch.empty((Bn, M, N), dtype=out_dtype, device=dev)
    if workspace is None and at == E2M1:
        workspace = torch.empty(max(gemm_workspace_size(Bn, M, N, K, at), 1), dtype=torch.uint8, device=dev)
    _check(lib().bsmm_gemm_atoms(Bn, M, N, K, _ptr(a), at, _ptr(b), bt, _ptr(a_atoms), _ptr(b_atoms),
                                 sc, _ptr(y), BF16 if y.dtype == torch.bfloat16 else F32,
                                 _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "bsmm_gemm_atoms")
    return y


def linear_backward_quantized(dy_n, dy_n_scales, w_t, w_t_scales, dy_t, dy_t_scales, x_t, x_t_scales,
                              fp8="e5m2", scales_are_atoms=False, dX=None, dW=None, workspace=None, stream=None):
    """The backward's two GEMMs from pre-quantized operands: dY along N
    [M, N], W^T [K, N], dY^T [N, M], X^T [K, M] with their scales (row-major,
    or atoms).  Returns ``(dX, dW)`` in bfloat16."""
    c = _code(fp8)
    _want(dy_n, "dy_n", itemsize=1)
    if dy_n.dim() != 2:
        raise ValueError("dy_n must be a 2-D code tensor [M, N]")
    M, N = dy_n.shape
    _want(w_t, "w_t", itemsize=1)
    if w_t.dim() != 2:
        raise ValueError("w_t must be a 2-D code tensor [K, N]")
    K = w_t.shape[0]
    # (codes, scales, rows, contraction) of each operand
    operands = (("dy_n", dy_n, dy_n_scales, M, N), ("w_t", w_t, w_t_scales, K, N),
                ("dy_t", dy_t, dy_t_scales, N, M), ("x_t", x_t, x_t_scales, K, M))
    for n, codes, scales, rows, kc in operands:
        _want(codes, n, (rows, kc), itemsize=1)
        if scales_are_atoms:
            _want(scales, f"{n}_scales", min_bytes=scale_atoms_size(1, rows, kc, c, SCALE_UE8M0))
        elif kc % 32 == 0:  # else the library says why
            _want(scales, f"{n}_scales", (rows, kc // 32), itemsize=1)
    bf16 = (torch.bfloat16,)
    if dX is not None:
        _want(dX, "dX", (M, K), dtypes=bf16)
    if dW is not None:
        _want(dW, "dW", (N, K), dtypes=bf16)
    if workspace is not None:
        _want(workspace, "workspace")
    dev = _on_device(dy_n=dy_n, dy_n_scales=dy_n_scales, w_t=w_t, w_t_scales=w_t_scales, dy_t=dy_t,
                     dy_t_scales=dy_t_scales, x_t=x_t, x_t_scales=x_t_scales, dX=dX, dW=dW, workspace=workspace)
    if dX is None:
        dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if dW is None:
        dW = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    need = lib().bsmm_linear_backward_quantized_workspace_size(M, N, K, 1 if scales_are_atoms else 0)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(lib().bsmm_linear_backward_quantized(M, N, K, c, _ptr(dy_n), _ptr(dy_n_scales), _ptr(w_t),
                                                _ptr(w_t_scales), _ptr(dy_t), _ptr(dy_t_scales), _ptr(x_t),
                                                _ptr(x_t_scales), 1 if scales_are_atoms else 0, _ptr(dX), _ptr(dW),
                                                _ptr(workspace), _nbytes(workspace),
                                                _stream(stream)), "bsmm_linear_backward_quantized")
    return dX, dW
