"""Host-side checks of the C-ABI library: it loads, exports every entry point
that include/h3q.h declares, and rejects bad arguments before touching a GPU.
No compute call is made here (these tests run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(h3q_\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def cdll():
    import w8a8_int8_linear_h3q_gb300 as h3q
    return h3q.load()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("h3q_quantize_weights", "h3q_quantize_act", "h3q_linear_w8a8",
                 "h3q_linear_workspace_bytes", "h3q_status_string", "h3q_version",
                 "h3q_workspace_status", "h3q_linear_w8a8_mma_sync"):
        assert must in names


def test_library_exports_every_declared_symbol(cdll):
    for name in _declared_functions():
        assert hasattr(cdll, name), name


def test_status_strings(cdll):
    import w8a8_int8_linear_h3q_gb300 as h3q
    for code in range(8):
        s = h3q.h3q_status_string(code)
        assert s and s != "unknown status"
    assert h3q.h3q_status_string(99) == "unknown status"
    assert h3q.h3q_version() >= 100


def test_workspace_size(cdll):
    import w8a8_int8_linear_h3q_gb300 as h3q
    assert h3q.h3q_linear_workspace_bytes(8192, 5376, 5376) >= 8192 * 5376 * 2
    assert h3q.h3q_linear_workspace_bytes(1, 1, 16) % 256 == 0


# Fake device addresses: aligned and non-null, never dereferenced because every
# call below is rejected on the host (argument checks come before any CUDA call).
A = ctypes.c_void_p(0x10000)
MIS = ctypes.c_void_p(0x10008)
NUL = None


def test_quantize_act_rejects_bad_args(cdll):
    q = cdll.h3q_quantize_act
    assert q(NUL, 4, 64, A, A, NUL) == 1                 # null input
    assert q(A, 4, 64, NUL, A, NUL) == 1                 # null output
    assert q(A, 0, 64, A, A, NUL) == 2                   # M = 0
    assert q(A, 4, 8, A, A, NUL) == 2                    # K < 16
    assert q(A, 4, 72, A, A, NUL) == 2                   # K % 16 != 0
    assert q(A, 4, 133152, A, A, NUL) == 2               # K past the INT32 bound
    assert q(MIS, 4, 64, A, A, NUL) == 3                 # misaligned
    assert q(A, 4, 64, A, MIS, NUL) == 3


def test_quantize_weights_rejects_bad_args(cdll):
    q = cdll.h3q_quantize_weights
    assert q(A, 2, 4, 64, A, A, NUL) == 1                # bad dtype
    assert q(NUL, 0, 4, 64, A, A, NUL) == 1
    assert q(A, 0, -1, 64, A, A, NUL) == 2
    assert q(A, 1, 4, 40, A, A, NUL) == 2
    assert q(A, 0, 4, 64, MIS, A, NUL) == 3


def test_linear_rejects_bad_args(cdll):
    f = cdll.h3q_linear_w8a8
    ws = cdll.h3q_linear_workspace_bytes(4, 8, 64)
    # x, xq, xs, wq, ws, bias, M, N, K, y, acc, workspace, bytes, stream
    assert f(A, A, NUL, A, A, NUL, 4, 8, 64, A, NUL, A, ws, NUL) == 1      # no xs
    assert f(A, A, A, A, A, NUL, 4, 8, 64, NUL, NUL, A, ws, NUL) == 1      # no output
    assert f(A, NUL, A, A, A, NUL, 4, 8, 64, A, NUL, NUL, 0, NUL) == 1     # no workspace
    assert f(NUL, NUL, A, A, A, NUL, 4, 8, 64, A, NUL, NUL, ws, NUL) == 1  # reuse, no workspace
    assert f(A, NUL, A, A, A, NUL, 4, 8, 64, A, NUL, A, ws - 256, NUL) == 1
    assert f(A, A, A, A, A, NUL, 4, 0, 64, A, NUL, A, ws, NUL) == 2        # N = 0
    assert f(A, A, A, A, A, NUL, 4, 8, 60, A, NUL, A, ws, NUL) == 2        # K % 16
    assert f(A, A, A, A, A, MIS, 4, 8, 64, A, NUL, A, ws, NUL) == 3        # misaligned bias
    assert f(A, A, A, A, A, NUL, 4, 8, 64, MIS, NUL, A, ws, NUL) == 3      # misaligned y


def test_status_and_legacy_entry_points_reject_bad_args(cdll):
    assert cdll.h3q_workspace_status(NUL, 4, 64, NUL) == 1
    assert cdll.h3q_workspace_status(MIS, 4, 64, NUL) == 3
    g = cdll.h3q_linear_w8a8_mma_sync
    # xq, xs, wq, ws, bias, M, N, K, y, acc, stream
    assert g(NUL, A, A, A, NUL, 4, 8, 64, A, NUL, NUL) == 1
    assert g(A, A, A, A, NUL, 4, 8, 64, NUL, NUL, NUL) == 1
    assert g(A, A, A, A, NUL, 4, 8, 24, A, NUL, NUL) == 2
    assert g(A, A, A, A, NUL, 4, 8, 64, MIS, NUL, NUL) == 3


def test_noalloc_scratch_bound_and_status_args(cdll):
    # the built-in scratch is 16 MiB: at N = K = 5376 it holds M = 1559 rows, not 1560
    assert cdll.h3q_linear_workspace_bytes(1559, 5376, 5376) <= 16 << 20
    assert cdll.h3q_linear_workspace_bytes(1560, 5376, 5376) > 16 << 20
    st = cdll.h3q_linear_w8a8_noalloc_status
    assert st(0, 5376, NUL) == 2                          # M < 1
    assert st(4, 8, NUL) == 2                             # K < 16
    assert st(4096, 5376, NUL) == 2                       # beyond the scratch
    f = cdll.h3q_linear_w8a8_noalloc
    # x, xq, xs, wq, ws, bias, M, N, K, y, acc, stream
    assert f(NUL, NUL, A, A, A, NUL, 4, 8, 64, A, NUL, NUL) == 1     # no x and no xq
    assert f(A, NUL, A, A, A, NUL, 4, 8, 64, NUL, NUL, NUL) == 1     # no output
    assert f(A, NUL, A, A, A, NUL, 4096, 128, 5376, A, NUL, NUL) == 2  # beyond the scratch


def test_valid_args_without_a_device_report_no_device(cdll):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: this checks the no-device report only")
    assert cdll.h3q_quantize_act(A, 4, 64, A, A, NUL) == 7
    # the no-alloc entry points check the device before looking up their scratch
    assert cdll.h3q_linear_w8a8_noalloc(A, NUL, A, A, A, NUL, 4, 8, 64, A, NUL, NUL) == 7
    assert cdll.h3q_linear_w8a8_noalloc_status(4, 64, NUL) == 7
    t = ctypes.c_double(-1.0)
    assert cdll.h3q_probe_mma_s8_tops(ctypes.byref(t), NUL) == 7
    assert t.value == 0.0
    t = ctypes.c_double(-1.0)
    assert cdll.h3q_probe_mma_f16_pair_tflops(ctypes.byref(t), 0, NUL) == 7
    assert t.value == 0.0


def test_grouped_linear_rejects_bad_args(cdll):
    f = cdll.h3q_linear_w8a8_grouped
    ws = cdll.h3q_linear_grouped_workspace_bytes(3, 4, 8, 64)
    assert cdll.h3q_linear_grouped_workspace_bytes(0, 4, 8, 64) == 0
    assert cdll.h3q_linear_grouped_workspace_bytes(5, 4, 8, 64) == 0
    assert (cdll.h3q_linear_grouped_workspace_bytes(3, 4096, 5376, 64)
            > cdll.h3q_linear_workspace_bytes(4096, 5376, 64))
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    P3 = arr(0x10000, 0x20000, 0x30000)
    one_null = arr(0x10000, None, 0x30000)
    one_mis = arr(0x10000, 0x10008, 0x30000)
    # x, xq, xs, G, wq, ws, bias, M, N, K, y, workspace, bytes, stream
    assert f(A, NUL, A, 0, P3, P3, NUL, 4, 8, 64, P3, A, ws, NUL) == 1         # G = 0
    assert f(A, NUL, A, 5, P3, P3, NUL, 4, 8, 64, P3, A, ws, NUL) == 1         # G = 5
    assert f(A, NUL, A, 3, NUL, P3, NUL, 4, 8, 64, P3, A, ws, NUL) == 1        # no weight array
    assert f(A, NUL, A, 3, one_null, P3, NUL, 4, 8, 64, P3, A, ws, NUL) == 1   # a NULL weight
    assert f(A, NUL, A, 3, P3, P3, NUL, 4, 8, 64, one_null, A, ws, NUL) == 1   # a NULL output
    assert f(A, NUL, NUL, 3, P3, P3, NUL, 4, 8, 64, P3, A, ws, NUL) == 1       # no xs
    assert f(A, NUL, A, 3, P3, P3, NUL, 4, 8, 64, P3, A, ws - 256, NUL) == 1   # workspace too small
    assert f(A, NUL, A, 3, P3, P3, NUL, 4, 8, 60, P3, A, ws, NUL) == 2         # K % 16
    assert f(A, NUL, A, 3, P3, one_mis, NUL, 4, 8, 64, P3, A, ws, NUL) == 3    # misaligned scale
    assert f(A, NUL, A, 3, P3, P3, one_mis, 4, 8, 64, P3, A, ws, NUL) == 3     # misaligned bias


def test_affine_entry_points_reject_bad_args(cdll):
    q = cdll.h3q_quantize_weights_affine
    # w, dtype, bits, N, K, q_out, ab_out, stream
    assert q(A, 2, 8, 4, 64, A, A, NUL) == 1             # bad dtype
    assert q(NUL, 0, 8, 4, 64, A, A, NUL) == 1           # null weights
    assert q(A, 0, 8, 4, 64, A, NUL, NUL) == 1           # null (step, offset) output
    for bits in (0, 2, 6, 16):
        assert q(A, 0, bits, 4, 64, A, A, NUL) == 1      # only 8 and 4 bits
    assert q(A, 0, 4, 4, 96, A, A, NUL) == 2             # K not a multiple of 64
    assert q(A, 0, 8, 0, 64, A, A, NUL) == 2             # N = 0
    assert q(A, 0, 8, 4, 64, MIS, A, NUL) == 3           # misaligned codes
    f = cdll.h3q_linear_affine_w8
    # x, q, ab, bias, M, N, K, y, status, stream
    assert f(NUL, A, A, NUL, 4, 8, 64, A, A, NUL) == 1   # null x
    assert f(A, A, A, NUL, 4, 8, 64, NUL, A, NUL) == 1   # null y
    assert f(A, A, A, NUL, 4, 8, 64, A, NUL, NUL) == 1   # null status word
    assert f(A, A, A, NUL, 4, 8, 80, A, A, NUL) == 2     # K % 64
    assert f(A, A, A, NUL, 0, 8, 64, A, A, NUL) == 2     # M = 0
    assert f(A, A, A, MIS, 4, 8, 64, A, A, NUL) == 3     # misaligned bias
    assert f(A, A, MIS, NUL, 4, 8, 64, A, A, NUL) == 3   # misaligned steps


def test_chunk_diagnostics_reject_bad_args(cdll):
    n = ctypes.c_int64(0)
    for fn in (cdll.h3q_linear_chunked_tiles, cdll.h3q_linear_checkpointed_tiles):
        assert fn(NUL, 4, 64, ctypes.byref(n), NUL) == 1
        assert fn(A, 4, 64, NUL, NUL) == 1
        assert fn(A, 0, 64, ctypes.byref(n), NUL) == 2
        assert fn(MIS, 4, 64, ctypes.byref(n), NUL) == 3


def test_probe_rejects_bad_args(cdll):
    assert cdll.h3q_probe_mma_s8_tops(NUL, NUL) == 1
    t = ctypes.c_double(0.0)
    assert cdll.h3q_probe_mma_f16_pair_tflops(NUL, 0, NUL) == 1
    assert cdll.h3q_probe_mma_f16_pair_tflops(ctypes.byref(t), 2, NUL) == 1
    assert cdll.h3q_probe_mma_f16_pair_tflops(ctypes.byref(t), -1, NUL) == 1


def test_selftest_rejects_bad_args(cdll):
    assert cdll.h3q_selftest_bounded_wait(NUL, NUL) == 1
    assert cdll.h3q_selftest_bounded_wait(ctypes.c_void_p(0x10002), NUL) == 3


def test_host_pipeline_rejects_bad_args(cdll):
    size = cdll.h3q_linear_w8a8_grouped_host_workspace_bytes
    ws = size(2, 100, 8, 64, 32)
    assert ws >= cdll.h3q_linear_grouped_workspace_bytes(2, 32, 8, 64)
    assert size(2, 100, 8, 64, 24) == 0                  # chunk rows not a multiple of 16
    assert size(2, 100, 8, 64, 0) == 0
    assert size(0, 100, 8, 64, 32) == 0                  # G outside 1..4
    assert size(5, 100, 8, 64, 32) == 0
    assert size(2, 0, 8, 64, 32) == 0
    # a chunk larger than M is sized for M rows
    assert size(2, 20, 8, 64, 4096) < size(2, 4096, 8, 64, 4096)
    f = cdll.h3q_linear_w8a8_grouped_host
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    P2 = arr(0x10000, 0x20000)
    one_null = arr(0x10000, None)
    one_mis = arr(0x10000, 0x10008)
    # x_host, G, wq, ws, bias, M, N, K, y_host, x_dev, xs, y_dev, chunk, first,
    # workspace, bytes, stream, h2d, d2h
    def call(x_host=A, G=2, wq=P2, sc=P2, bias=NUL, M=100, N=8, K=64, y_host=P2, x_dev=A,
             xs=A, y_dev=P2, chunk=32, first=0, work=A, nbytes=ws):
        return f(x_host, G, wq, sc, bias, M, N, K, y_host, x_dev, xs, y_dev, chunk, first,
                 work, nbytes, NUL, NUL, NUL)
    assert call(G=0) == 1
    assert call(G=5) == 1
    assert call(x_host=NUL) == 1
    assert call(y_host=NUL) == 1
    assert call(y_host=one_null) == 1                    # a NULL host output
    assert call(y_dev=one_null) == 1                     # a NULL device output
    assert call(wq=one_null) == 1
    assert call(xs=NUL) == 1
    assert call(work=NUL) == 1
    assert call(chunk=24) == 1                           # chunk rows not a multiple of 16
    assert call(first=8) == 1                            # first chunk not a multiple of 16
    assert call(first=48) == 1                           # first chunk above the steady size
    assert call(nbytes=ws - 256) == 1                    # workspace too small
    assert call(K=60) == 2                               # K % 16
    assert call(M=0) == 2
    assert call(x_host=MIS) == 3
    assert call(y_dev=one_mis) == 3
    assert call(y_host=one_mis) == 3
    assert call(xs=MIS) == 3


def test_host_pipeline_without_a_device_reports_no_device(cdll):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: this checks the no-device report only")
    P2 = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    ws = cdll.h3q_linear_w8a8_grouped_host_workspace_bytes(2, 100, 8, 64, 32)
    assert cdll.h3q_linear_w8a8_grouped_host(A, 2, P2, P2, NUL, 100, 8, 64, P2, A, A, P2, 32,
                                             16, A, ws, NUL, NUL, NUL) == 7


@pytest.mark.parametrize("M,chunk,first", [(8192, 2048, 0), (8192, 1024, 256), (77, 16, 16),
                                           (1000, 256, 64), (5, 2048, 0), (2048, 2048, 2048),
                                           (75647, 4096, 16), (1, 16, 0)])
def test_host_pipeline_chunk_plan(cdll, M, chunk, first):
    # the plan the pinned-host pipeline follows: it covers M exactly; chunks
    # ramp from the first size by doubling up to the steady size; every chunk
    # but the last is a multiple of 16 rows (so each chunk's row blocks stay
    # 16-byte aligned); and the count fits the workspace's status slots
    import w8a8_int8_linear_h3q_gb300 as h3q
    rows = h3q.h3q_linear_w8a8_grouped_host_chunks(M, chunk, first)
    assert sum(rows) == M and all(r >= 1 for r in rows)
    f = first or max(16, -(-(chunk // 4) // 16) * 16)
    want, r = [], f
    while sum(want) < M:
        want.append(min(r, M - sum(want)))
        r = min(2 * r, chunk)
    assert rows == want
    assert all(r % 16 == 0 for r in rows[:-1])
    slots = len(rows) * 4
    call = cdll.h3q_linear_grouped_workspace_bytes(2, min(chunk, M), 8, 64)
    assert cdll.h3q_linear_w8a8_grouped_host_workspace_bytes(2, M, 8, 64, chunk) >= call + slots


def test_host_pipeline_chunk_plan_rejects_bad_args(cdll):
    import w8a8_int8_linear_h3q_gb300 as h3q
    f = cdll.h3q_linear_w8a8_grouped_host_chunks
    assert f(0, 32, 0, None, 0) == -1                    # M = 0
    assert f(100, 24, 0, None, 0) == -1                  # chunk not a multiple of 16
    assert f(100, 32, 8, None, 0) == -1                  # first not a multiple of 16
    assert f(100, 32, 48, None, 0) == -1                 # first above the steady size
    assert f(100, 32, 0, None, 0) == 4                   # count only: 16, 32, 32, 20
    with pytest.raises(ValueError):
        h3q.h3q_linear_w8a8_grouped_host_chunks(100, 24)


def test_binding_checks_tensors_before_any_device_work():
    """The Python binding's argument checks (one combined test per tensor)
    reject host tensors where device tensors are required, with the error
    naming the argument, before the library is asked to do anything."""
    torch = pytest.importorskip("torch")
    import w8a8_int8_linear_h3q_gb300 as h3q
    wq = [torch.zeros((64, 64), dtype=torch.int8)]
    ws = [torch.ones((64,), dtype=torch.float32)]
    with pytest.raises(TypeError, match="wq must be a CUDA tensor"):
        h3q.GroupedHostCall(torch.zeros((64, 64), dtype=torch.bfloat16), wq, ws)
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        h3q._need(torch.zeros((4,), dtype=torch.float32), torch.float32, (4,), "xs")
    with pytest.raises(TypeError, match="page-locked"):
        h3q._need_pinned(torch.zeros((4,), dtype=torch.float32), torch.float32, (4,), "x_host")
