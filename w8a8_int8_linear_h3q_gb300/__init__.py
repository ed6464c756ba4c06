"""Python binding of libh3q.so: the GB300 (sm_103a) W8A8 INT8 projection Linear.

The functions carry the C entry points' names (include/h3q.h) and only
marshal arguments: torch tensors supply device memory and the current CUDA
stream, and every step of the computation runs in the library's kernels.
There is no CPU or library fallback: if libh3q.so cannot be built or loaded,
``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

H3Q_OK = 0
H3Q_ERR_INVALID_ARG = 1
H3Q_ERR_UNSUPPORTED_SHAPE = 2
H3Q_ERR_MISALIGNED = 3
H3Q_ERR_NONFINITE = 4
H3Q_ERR_CUDA = 5
H3Q_ERR_TIMEOUT = 6
H3Q_ERR_NO_DEVICE = 7
H3Q_DTYPE_F32 = 0
H3Q_DTYPE_BF16 = 1

_lib = None


class H3QError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {h3q_status_string(status)} (status {status})")


def _declare(lib):
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.h3q_status_string.argtypes = [i32]
    lib.h3q_status_string.restype = ctypes.c_char_p
    lib.h3q_version.argtypes = []
    lib.h3q_version.restype = i32
    lib.h3q_quantize_weights.argtypes = [vp, i32, i64, i64, vp, vp, vp]
    lib.h3q_quantize_weights.restype = i32
    lib.h3q_quantize_act.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.h3q_quantize_act.restype = i32
    lib.h3q_linear_workspace_bytes.argtypes = [i64, i64, i64]
    lib.h3q_linear_workspace_bytes.restype = sz
    lib.h3q_linear_w8a8.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, vp, vp, sz, vp]
    lib.h3q_linear_w8a8.restype = i32
    lib.h3q_workspace_status.argtypes = [vp, i64, i64, vp]
    lib.h3q_workspace_status.restype = i32
    lib.h3q_linear_grouped_workspace_bytes.argtypes = [i32, i64, i64, i64]
    lib.h3q_linear_grouped_workspace_bytes.restype = sz
    lib.h3q_linear_w8a8_grouped.argtypes = [vp, vp, vp, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                            ctypes.POINTER(vp), i64, i64, i64, ctypes.POINTER(vp),
                                            vp, sz, vp]
    lib.h3q_linear_w8a8_grouped.restype = i32
    lib.h3q_linear_w8a8_grouped_host_workspace_bytes.argtypes = [i32, i64, i64, i64, i64]
    lib.h3q_linear_w8a8_grouped_host_workspace_bytes.restype = sz
    lib.h3q_linear_w8a8_grouped_host_chunks.argtypes = [i64, i64, i64, ctypes.POINTER(i64), i64]
    lib.h3q_linear_w8a8_grouped_host_chunks.restype = i64
    lib.h3q_linear_w8a8_grouped_host.argtypes = [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                 ctypes.POINTER(vp), i64, i64, i64,
                                                 ctypes.POINTER(vp), vp, vp, ctypes.POINTER(vp),
                                                 i64, i64, vp, sz, vp, vp, vp]
    lib.h3q_linear_w8a8_grouped_host.restype = i32
    lib.h3q_linear_chunked_tiles.argtypes = [vp, i64, i64, ctypes.POINTER(i64), vp]
    lib.h3q_linear_chunked_tiles.restype = i32
    lib.h3q_linear_checkpointed_tiles.argtypes = [vp, i64, i64, ctypes.POINTER(i64), vp]
    lib.h3q_linear_checkpointed_tiles.restype = i32
    lib.h3q_linear_w8a8_mma_sync.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp, vp, vp]
    lib.h3q_linear_w8a8_mma_sync.restype = i32
    lib.h3q_linear_w8a8_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, vp, vp]
    lib.h3q_linear_w8a8_noalloc.restype = i32
    lib.h3q_probe_mma_s8_tops.argtypes = [ctypes.POINTER(ctypes.c_double), vp]
    lib.h3q_probe_mma_s8_tops.restype = i32
    lib.h3q_probe_mma_f16_pair_tflops.argtypes = [ctypes.POINTER(ctypes.c_double), i32, vp]
    lib.h3q_probe_mma_f16_pair_tflops.restype = i32
    lib.h3q_linear_w8a8_noalloc_status.argtypes = [i64, i64, vp]
    lib.h3q_linear_w8a8_noalloc_status.restype = i32
    lib.h3q_selftest_bounded_wait.argtypes = [vp, vp]
    lib.h3q_selftest_bounded_wait.restype = i32
    lib.h3q_quantize_weights_affine.argtypes = [vp, i32, i32, i64, i64, vp, vp, vp]
    lib.h3q_quantize_weights_affine.restype = i32
    lib.h3q_linear_affine_w8.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, vp]
    lib.h3q_linear_affine_w8.restype = i32
    return lib


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libh3q.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is None:
        if build_if_missing and _build.stale():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libh3q.so is missing at {_build.LIB}; build it with "
                               "python -m w8a8_int8_linear_h3q_gb300._build")
        _lib = _declare(ctypes.CDLL(_build.LIB))
    return _lib


def lib_path() -> str:
    return _build.LIB


# --- marshalling helpers ------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_torch = None


def _tm():
    """torch, imported on first use (the checks below run on every call, so
    they keep their per-tensor cost to one combined test)."""
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def _stream(stream):
    s = _tm().cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, shape, name):
    torch = _tm()
    if (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype is dtype and t.is_contiguous()
            and (shape is None or t.shape == tuple(shape))):
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _need_pinned(t, dtype, shape, name):
    torch = _tm()
    if (isinstance(t, torch.Tensor) and not t.is_cuda and t.dtype is dtype
            and t.is_contiguous() and (shape is None or t.shape == tuple(shape))
            and t.is_pinned()):
        return
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
        raise TypeError(f"{name} must be a page-locked (pinned) CPU tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check(status, where):
    if status != H3Q_OK:
        raise H3QError(status, where)


# --- the entry points --------------------------------------------------------------

def h3q_status_string(status: int) -> str:
    return load().h3q_status_string(int(status)).decode()


def h3q_version() -> int:
    return int(load().h3q_version())


def h3q_linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().h3q_linear_workspace_bytes(M, N, K))


def h3q_quantize_weights(w, q_out=None, scale_out=None, stream=None):
    """A1: FP32 or BF16 weight [N, K] -> (int8 [N, K], FP32 scale [N]).  Synchronises."""
    import torch
    if w.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("weights must be float32 or bfloat16")
    _need(w, w.dtype, None, "w")
    N, K = w.shape
    q_out = torch.empty((N, K), dtype=torch.int8, device=w.device) if q_out is None else q_out
    scale_out = torch.empty((N,), dtype=torch.float32, device=w.device) if scale_out is None else scale_out
    _need(q_out, torch.int8, (N, K), "q_out")
    _need(scale_out, torch.float32, (N,), "scale_out")
    dt = H3Q_DTYPE_F32 if w.dtype == torch.float32 else H3Q_DTYPE_BF16
    _check(load().h3q_quantize_weights(_ptr(w), dt, N, K, _ptr(q_out), _ptr(scale_out),
                                       _stream(stream)), "h3q_quantize_weights")
    return q_out, scale_out


def h3q_quantize_weights_affine(w, q_out=None, ab_out=None, stream=None, bits=8):
    """The group-wise affine comparison scheme, offline: FP32 or BF16 weight
    [N, K] (K a multiple of 64) -> (uint8 codes [N, K] in [0, 2^bits - 1], FP32
    (step, offset) pairs [N, K/64, 2]); bits 8 (Q8/g64) or 4 (Q4/g64, one code
    per byte).  Synchronises."""
    import torch
    if w.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("weights must be float32 or bfloat16")
    _need(w, w.dtype, None, "w")
    N, K = w.shape
    q_out = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q_out is None else q_out
    ab_out = (torch.empty((N, K // 64, 2), dtype=torch.float32, device=w.device)
              if ab_out is None else ab_out)
    _need(q_out, torch.uint8, (N, K), "q_out")
    _need(ab_out, torch.float32, (N, K // 64, 2), "ab_out")
    dt = H3Q_DTYPE_F32 if w.dtype == torch.float32 else H3Q_DTYPE_BF16
    _check(load().h3q_quantize_weights_affine(_ptr(w), dt, bits, N, K, _ptr(q_out),
                                              _ptr(ab_out), _stream(stream)),
           "h3q_quantize_weights_affine")
    return q_out, ab_out


def h3q_linear_affine_w8(x, q, ab, bias=None, *, y=None, status=None, stream=None):
    """The comparison scheme's weight-only Linear: BF16 x [M, K] against the
    dequantised codes.  Returns {"y": BF16 [M, N], "status": int32 [1]} (the
    status word is nonzero after the call if a device-side wait gave up)."""
    import torch
    _need(x, torch.bfloat16, None, "x")
    _need(q, torch.uint8, None, "q")
    M, K = x.shape
    N = q.shape[0]
    if q.shape[1] != K:
        raise ValueError("x and q disagree on K")
    _need(ab, torch.float32, (N, K // 64, 2), "ab")
    if bias is not None:
        _need(bias, torch.bfloat16, (N,), "bias")
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    _need(y, torch.bfloat16, (M, N), "y")
    status = torch.empty((4,), dtype=torch.int32, device=x.device) if status is None else status
    _check(load().h3q_linear_affine_w8(_ptr(x), _ptr(q), _ptr(ab), _ptr(bias), M, N, K, _ptr(y),
                                       _ptr(status), _stream(stream)), "h3q_linear_affine_w8")
    return {"y": y, "status": status}


def h3q_selftest_bounded_wait(status=None, stream=None) -> int:
    """Drive a device-side bounded wait to its limit (about 2 s).  Returns the
    status code: H3Q_ERR_TIMEOUT is the expected, healthy result."""
    import torch
    if status is None:
        status = torch.empty((4,), dtype=torch.int32, device="cuda")
    return int(load().h3q_selftest_bounded_wait(_ptr(status), _stream(stream)))


def h3q_probe_mma_s8_tops(stream=None) -> float:
    """Measured rate (TOPS) of the legacy mma.sync m16n8k32 s8 instruction,
    the one INT8 tensor instruction of sm_103.  Synchronises; about 40 ms."""
    t = ctypes.c_double(0.0)
    _check(load().h3q_probe_mma_s8_tops(ctypes.byref(t), _stream(stream)),
           "h3q_probe_mma_s8_tops")
    return float(t.value)


def h3q_probe_mma_f16_pair_tflops(a_in_smem: bool = False, stream=None) -> float:
    """Measured rate (TFLOP/s) of tcgen05.mma.cta_group::2.kind::f16 at
    M = N = 256, K = 16, the instruction of the hot GEMM: A in TMEM (the
    kernel's form) or, with a_in_smem, in shared memory.  Synchronises;
    about 4 ms."""
    t = ctypes.c_double(0.0)
    _check(load().h3q_probe_mma_f16_pair_tflops(ctypes.byref(t), 1 if a_in_smem else 0,
                                                _stream(stream)),
           "h3q_probe_mma_f16_pair_tflops")
    return float(t.value)


def h3q_quantize_act(x, q_out=None, scale_out=None, stream=None):
    """A2: BF16 activations [M, K] -> (int8 [M, K], FP32 scale [M])."""
    import torch
    _need(x, torch.bfloat16, None, "x")
    M, K = x.shape
    q_out = torch.empty((M, K), dtype=torch.int8, device=x.device) if q_out is None else q_out
    scale_out = torch.empty((M,), dtype=torch.float32, device=x.device) if scale_out is None else scale_out
    _need(q_out, torch.int8, (M, K), "q_out")
    _need(scale_out, torch.float32, (M,), "scale_out")
    _check(load().h3q_quantize_act(_ptr(x), M, K, _ptr(q_out), _ptr(scale_out), _stream(stream)),
           "h3q_quantize_act")
    return q_out, scale_out


def h3q_linear_w8a8(x, wq, ws, bias=None, *, xq=None, xs=None, y=None, acc_out=None,
                    want_y=True, want_acc=False, want_xq=False, workspace=None, M=None,
                    stream=None):
    """A2 + A3 + A4.  ``x`` BF16 [M, K]; or None with ``xq``/``xs`` given
    (pre-quantised); or None with ``xq`` None (reuse: ``workspace`` still holds
    the coded activations of the previous call on it; pass ``xs`` and ``M``).

    Returns a dict with whichever of ``y`` (BF16 [M, N]), ``acc`` (int32 [M, N]),
    ``xq`` (int8 [M, K]) and ``xs`` (FP32 [M]) were produced, and the
    ``workspace`` used.  Outputs and the workspace are allocated here when not
    given (allocation is plumbing; the library itself allocates nothing).
    """
    import torch
    _need(wq, torch.int8, None, "wq")
    N, K = wq.shape
    dev = wq.device
    if x is not None:
        _need(x, torch.bfloat16, None, "x")
        M = x.shape[0]
        if x.shape[1] != K:
            raise ValueError("x and wq disagree on K")
        if want_xq and xq is None:
            xq = torch.empty((M, K), dtype=torch.int8, device=dev)
        if xs is None:
            xs = torch.empty((M,), dtype=torch.float32, device=dev)
    elif xq is not None:
        if xs is None:
            raise ValueError("pre-quantised call needs xs")
        M = xq.shape[0]
    else:
        if xs is None or workspace is None:
            raise ValueError("reuse call needs xs and the workspace")
        M = xs.shape[0]
    if xq is not None:
        _need(xq, torch.int8, (M, K), "xq")
    _need(xs, torch.float32, (M,), "xs")
    _need(ws, torch.float32, (N,), "ws")
    if bias is not None:
        _need(bias, torch.bfloat16, (N,), "bias")
    if want_y and y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if want_acc and acc_out is None:
        acc_out = torch.empty((M, N), dtype=torch.int32, device=dev)
    if y is not None:
        _need(y, torch.bfloat16, (M, N), "y")
    if acc_out is not None:
        _need(acc_out, torch.int32, (M, N), "acc_out")
    need = h3q_linear_workspace_bytes(M, N, K)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    _check(load().h3q_linear_w8a8(_ptr(x), _ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), _ptr(bias),
                                  M, N, K, _ptr(y), _ptr(acc_out), _ptr(workspace), wbytes,
                                  _stream(stream)), "h3q_linear_w8a8")
    out = {"xs": xs, "workspace": workspace}
    if y is not None:
        out["y"] = y
    if acc_out is not None:
        out["acc"] = acc_out
    if xq is not None:
        out["xq"] = xq
    return out


def h3q_workspace_status(workspace, M: int, K: int, stream=None) -> int:
    """Status word of the last linear call on ``workspace``: 0 = ok,
    H3Q_ERR_TIMEOUT if a bounded device-side wait gave up.  Synchronises."""
    return int(load().h3q_workspace_status(_ptr(workspace), M, K, _stream(stream)))


def h3q_linear_grouped_workspace_bytes(G: int, M: int, N: int, K: int) -> int:
    return int(load().h3q_linear_grouped_workspace_bytes(G, M, N, K))


def h3q_linear_w8a8_grouped(x, wqs, wss, biases=None, *, xq=None, xs=None, ys=None,
                            workspace=None, M=None, stream=None):
    """A2 once + A3 + A4 for the Linears (wqs[g], wss[g], biases[g]) that share
    the input, in one GEMM launch.  ``x`` BF16 [M, K], or None with ``xq``/``xs``
    (pre-quantised), or None with ``xq`` None (reuse: pass ``xs``, ``M`` and the
    ``workspace`` of an earlier call).  Returns a dict with the outputs ``ys``
    (BF16 [M, N] each), ``xs`` and the ``workspace``."""
    import torch
    G = len(wqs)
    if not 1 <= G <= 4 or len(wss) != G or (biases is not None and len(biases) != G):
        raise ValueError("1..4 Linears, with one scale vector (and bias) each")
    for w in wqs:
        _need(w, torch.int8, tuple(wqs[0].shape), "wq")
    N, K = wqs[0].shape
    dev = wqs[0].device
    if x is not None:
        _need(x, torch.bfloat16, None, "x")
        M = x.shape[0]
        if xs is None:
            xs = torch.empty((M,), dtype=torch.float32, device=dev)
    elif xq is not None:
        if xs is None:
            raise ValueError("pre-quantised call needs xs")
        M = xq.shape[0]
        _need(xq, torch.int8, (M, K), "xq")
    else:
        if xs is None or workspace is None:
            raise ValueError("reuse call needs xs and the workspace")
        M = xs.shape[0]
    _need(xs, torch.float32, (M,), "xs")
    for s in wss:
        _need(s, torch.float32, (N,), "ws")
    if biases is not None:
        for b in biases:
            if b is not None:
                _need(b, torch.bfloat16, (N,), "bias")
    if ys is None:
        ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(G)]
    for y in ys:
        _need(y, torch.bfloat16, (M, N), "y")
    need = h3q_linear_grouped_workspace_bytes(G, M, N, K)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    arr = lambda ts: (ctypes.c_void_p * G)(*[None if t is None else t.data_ptr() for t in ts])
    _check(load().h3q_linear_w8a8_grouped(
        _ptr(x), _ptr(xq), _ptr(xs), G, arr(wqs), arr(wss),
        None if biases is None else arr(biases), M, N, K, arr(ys), _ptr(workspace), wbytes,
        _stream(stream)), "h3q_linear_w8a8_grouped")
    return {"ys": ys, "xs": xs, "workspace": workspace}


def h3q_linear_w8a8_grouped_host_workspace_bytes(G: int, M: int, N: int, K: int,
                                                 chunk_rows: int) -> int:
    return int(load().h3q_linear_w8a8_grouped_host_workspace_bytes(G, M, N, K, chunk_rows))


def h3q_linear_w8a8_grouped_host_chunks(M: int, chunk_rows: int = 2048, first_rows: int = 0) -> list:
    """Sizes of the row chunks h3q_linear_w8a8_grouped_host makes of M rows."""
    lib = load()
    n = int(lib.h3q_linear_w8a8_grouped_host_chunks(M, chunk_rows, first_rows, None, 0))
    if n < 0:
        raise ValueError("chunk_rows must be a positive multiple of 16 and first_rows 0 or a "
                         "multiple of 16 in [16, chunk_rows]; M >= 1")
    out = (ctypes.c_int64 * n)()
    lib.h3q_linear_w8a8_grouped_host_chunks(M, chunk_rows, first_rows, out, n)
    return list(out)


class GroupedHostCall:
    """h3q_linear_w8a8_grouped_host with its arguments checked, its buffers
    allocated and its C arguments marshalled once; calling the object runs
    the call again on the same tensors.  For repeated steps: write the next
    step's X into ``x_host`` (it is read at each call) and call.  Every call
    still uploads X, runs the grouped Linear and downloads the outputs, and
    synchronises.  The object keeps its tensors alive."""

    def __init__(self, x_host, wqs, wss, biases=None, *, ys_host=None, x_dev=None, xs=None,
                 ys_dev=None, chunk_rows=2048, first_rows=0, workspace=None, stream=None,
                 h2d_stream=None, d2h_stream=None):
        torch = _tm()
        G = len(wqs)
        if not 1 <= G <= 4 or len(wss) != G or (biases is not None and len(biases) != G):
            raise ValueError("1..4 Linears, with one scale vector (and bias) each")
        for w in wqs:
            _need(w, torch.int8, tuple(wqs[0].shape), "wq")
        N, K = wqs[0].shape
        dev = wqs[0].device
        _need_pinned(x_host, torch.bfloat16, None, "x_host")
        M = x_host.shape[0]
        if x_host.shape[1] != K:
            raise ValueError("x_host and wq disagree on K")
        for sc in wss:
            _need(sc, torch.float32, (N,), "ws")
        if biases is not None:
            for b in biases:
                if b is not None:
                    _need(b, torch.bfloat16, (N,), "bias")
        if ys_host is None:   # one [G, M, N] buffer: a chunk's downloads are then one copy
            yh = torch.empty((G, M, N), dtype=torch.bfloat16).pin_memory()
            ys_host = [yh[g] for g in range(G)]
        for y in ys_host:
            _need_pinned(y, torch.bfloat16, (M, N), "y_host")
        if x_dev is None:
            x_dev = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        if xs is None:
            xs = torch.empty((M,), dtype=torch.float32, device=dev)
        if ys_dev is None:
            yd = torch.empty((G, M, N), dtype=torch.bfloat16, device=dev)
            ys_dev = [yd[g] for g in range(G)]
        _need(x_dev, torch.bfloat16, (M, K), "x_dev")
        _need(xs, torch.float32, (M,), "xs")
        for y in ys_dev:
            _need(y, torch.bfloat16, (M, N), "y_dev")
        need = h3q_linear_w8a8_grouped_host_workspace_bytes(G, M, N, K, chunk_rows)
        if workspace is None:
            workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
        wbytes = workspace.numel() * workspace.element_size()
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        if h2d_stream is None:
            h2d_stream = torch.cuda.Stream(dev)
        if d2h_stream is None:
            d2h_stream = torch.cuda.Stream(dev)
        arr = lambda ts: (ctypes.c_void_p * G)(*[None if t is None else t.data_ptr() for t in ts])
        self._keep = (x_host, list(wqs), list(wss), biases, ys_host, x_dev, xs, ys_dev, workspace,
                      stream, h2d_stream, d2h_stream)
        self._args = (_ptr(x_host), G, arr(wqs), arr(wss), None if biases is None else arr(biases),
                      M, N, K, arr(ys_host), _ptr(x_dev), _ptr(xs), arr(ys_dev), chunk_rows,
                      first_rows, _ptr(workspace), wbytes, _stream(stream), _stream(h2d_stream),
                      _stream(d2h_stream))
        self._fn = load().h3q_linear_w8a8_grouped_host
        self.ys = ys_host
        self.ys_dev, self.x_dev, self.xs, self.workspace = ys_dev, x_dev, xs, workspace

    def __call__(self):
        _check(self._fn(*self._args), "h3q_linear_w8a8_grouped_host")
        return self.ys


def h3q_linear_w8a8_grouped_host(x_host, wqs, wss, biases=None, *, ys_host=None, x_dev=None,
                                 xs=None, ys_dev=None, chunk_rows=2048, first_rows=0,
                                 workspace=None, stream=None, h2d_stream=None, d2h_stream=None):
    """The grouped Linear from and to page-locked host memory: ``x_host`` is a
    pinned CPU BF16 tensor [M, K]; the outputs ``ys`` are pinned CPU BF16
    tensors [M, N].  X goes up and the outputs come down in row chunks that
    overlap the copies with the grouped calls (on ``stream``; the copies on
    ``h2d_stream`` and ``d2h_stream``).  Device staging (``x_dev``, ``xs``,
    ``ys_dev``), the workspace, the host outputs and the copy streams are
    allocated here when not given.  Synchronises.  Returns a dict with ``ys``
    (host), ``ys_dev``, ``x_dev``, ``xs`` and the ``workspace``.  (For repeated
    calls on the same tensors, GroupedHostCall checks and marshals once.)"""
    c = GroupedHostCall(x_host, wqs, wss, biases, ys_host=ys_host, x_dev=x_dev, xs=xs,
                        ys_dev=ys_dev, chunk_rows=chunk_rows, first_rows=first_rows,
                        workspace=workspace, stream=stream, h2d_stream=h2d_stream,
                        d2h_stream=d2h_stream)
    c()
    return {"ys": c.ys, "ys_dev": c.ys_dev, "x_dev": c.x_dev, "xs": c.xs,
            "workspace": c.workspace}


def h3q_linear_chunked_tiles(workspace, M: int, K: int, stream=None) -> int:
    """Tiles (128 tokens x 256 channels) that the last linear call on
    ``workspace`` computed in K chunks.  Synchronises."""
    n = ctypes.c_int64(-1)
    _check(load().h3q_linear_chunked_tiles(_ptr(workspace), M, K, ctypes.byref(n),
                                           _stream(stream)), "h3q_linear_chunked_tiles")
    return int(n.value)


def h3q_linear_checkpointed_tiles(workspace, M: int, K: int, stream=None) -> int:
    """Tiles (256 tokens x 256 channels) that the last linear call on
    ``workspace`` kept on one accumulator by way of checkpoints.  Synchronises."""
    n = ctypes.c_int64(-1)
    _check(load().h3q_linear_checkpointed_tiles(_ptr(workspace), M, K, ctypes.byref(n),
                                                _stream(stream)), "h3q_linear_checkpointed_tiles")
    return int(n.value)


def h3q_linear_w8a8_mma_sync(xq, xs, wq, ws, bias=None, *, y=None, acc_out=None, want_y=True,
                             want_acc=False, stream=None):
    """A3 + A4 from pre-quantised activations on the legacy mma.sync INT8 path."""
    import torch
    _need(xq, torch.int8, None, "xq")
    _need(wq, torch.int8, None, "wq")
    M, K = xq.shape
    N = wq.shape[0]
    if wq.shape[1] != K:
        raise ValueError("xq and wq disagree on K")
    _need(xs, torch.float32, (M,), "xs")
    _need(ws, torch.float32, (N,), "ws")
    if bias is not None:
        _need(bias, torch.bfloat16, (N,), "bias")
    if want_y and y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    if want_acc and acc_out is None:
        acc_out = torch.empty((M, N), dtype=torch.int32, device=xq.device)
    _check(load().h3q_linear_w8a8_mma_sync(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), _ptr(bias),
                                           M, N, K, _ptr(y), _ptr(acc_out), _stream(stream)),
           "h3q_linear_w8a8_mma_sync")
    out = {}
    if y is not None:
        out["y"] = y
    if acc_out is not None:
        out["acc"] = acc_out
    return out


def h3q_linear_w8a8_noalloc(x, wq, ws, bias=None, *, xq=None, xs=None, y=None, acc_out=None,
                            want_y=True, want_acc=False, stream=None):
    """As h3q_linear_w8a8, with the scratch built into the library (no workspace).

    For callers that cannot allocate device memory at call time; shapes whose
    workspace would exceed 16 MiB are rejected.  ``x`` BF16 [M, K], or None
    with ``xq``/``xs`` given.  Output tensors are allocated here when not given.
    """
    import torch
    _need(wq, torch.int8, None, "wq")
    N, K = wq.shape
    dev = wq.device
    if x is not None:
        _need(x, torch.bfloat16, None, "x")
        M = x.shape[0]
        if xs is None:
            xs = torch.empty((M,), dtype=torch.float32, device=dev)
    else:
        if xq is None or xs is None:
            raise ValueError("without x, both xq and xs are needed")
        M = xq.shape[0]
    if xq is not None:
        _need(xq, torch.int8, (M, K), "xq")
    _need(xs, torch.float32, (M,), "xs")
    _need(ws, torch.float32, (N,), "ws")
    if bias is not None:
        _need(bias, torch.bfloat16, (N,), "bias")
    if want_y and y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if want_acc and acc_out is None:
        acc_out = torch.empty((M, N), dtype=torch.int32, device=dev)
    _check(load().h3q_linear_w8a8_noalloc(_ptr(x), _ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws),
                                          _ptr(bias), M, N, K, _ptr(y), _ptr(acc_out),
                                          _stream(stream)), "h3q_linear_w8a8_noalloc")
    out = {"xs": xs}
    if y is not None:
        out["y"] = y
    if acc_out is not None:
        out["acc"] = acc_out
    return out


def h3q_linear_w8a8_noalloc_status(M: int, K: int, stream=None) -> int:
    """Status word of the last h3q_linear_w8a8_noalloc (same M and K) on the
    current device: 0 = ok, H3Q_ERR_TIMEOUT if a bounded device-side wait gave
    up.  Synchronises."""
    return int(load().h3q_linear_w8a8_noalloc_status(M, K, _stream(stream)))
