"""Guard bands around every buffer the library writes (the substitute for a
memory checker, which this GPU pool does not offer).

Each output -- y, the raw INT32 accumulators, the INT8 activations and their
scales, every output of a grouped call, the host pipeline's device staging --
is carved out of a larger allocation with 4 KiB of a known byte pattern on
both sides, and the workspace gets the pattern past the size the library asks
for.  After ragged calls (M, N and K chosen to leave partial tiles, vectors and
k-blocks) every guard byte must still hold the pattern: a tail store or a
TMA/vector access that runs past a buffer would change one.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


class Guarded:
    """A tensor of `shape` and `dtype` placed between two guard bands."""

    def __init__(self, shape, dtype, dev, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = n
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device=dev)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _operands(M, N, K, seed, dev):
    c = synth.make_linear(M, N, K, seed=seed, outlier_p=0.01, outlier_mul=20.0)
    x = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    w = torch.from_numpy(c.w[0]).to(dev)
    b = torch.from_numpy(c.bias_bits[0].view(np.int16)).view(torch.bfloat16).to(dev)
    return x, w, b


# odd N keeps 2-byte output stores; even N takes the paired 4-byte stores, whose last pair
# ends exactly at the row's end (256 x 130, 1024 x 5382)
SHAPES = [(1, 1, 16), (127, 131, 16), (129, 257, 1040), (255, 1, 1040), (257, 131, 5376),
          (1, 5383, 5376), (129, 5383, 1040), (257, 257, 5376), (32767, 131, 1040),
          (32767, 5383, 5376), (256, 130, 1040), (1024, 5382, 5376)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_writes_stay_inside_their_buffers(lib, dev, M, N, K):
    x, w, b = _operands(M, N, K, seed=M + 3 * N + 7 * K, dev=dev)
    qw = Guarded((N, K), torch.int8, dev)
    sw = Guarded((N,), torch.float32, dev)
    lib.h3q_quantize_weights(w, q_out=qw.t, scale_out=sw.t)
    y = Guarded((M, N), torch.bfloat16, dev)
    acc = Guarded((M, N), torch.int32, dev)
    xq = Guarded((M, K), torch.int8, dev)
    xs = Guarded((M,), torch.float32, dev)
    need = lib.h3q_linear_workspace_bytes(M, N, K)
    ws = Guarded((need,), torch.uint8, dev)
    # quantise from BF16, then reuse the coded activations, then pre-quantised
    lib.h3q_linear_w8a8(x, qw.t, sw.t, b, xq=xq.t, xs=xs.t, y=y.t, acc_out=acc.t,
                        workspace=ws.t)
    lib.h3q_linear_w8a8(None, qw.t, sw.t, b, xs=xs.t, y=y.t, acc_out=acc.t, workspace=ws.t)
    lib.h3q_linear_w8a8(None, qw.t, sw.t, b, xq=xq.t, xs=xs.t, y=y.t, workspace=ws.t)
    torch.cuda.synchronize()
    for name, g in (("q_w", qw), ("s_w", sw), ("y", y), ("acc", acc), ("xq", xq), ("xs", xs),
                    ("workspace", ws)):
        assert g.intact(), f"{name}: a guard byte changed ({M}x{N}x{K})"
    assert lib.h3q_workspace_status(ws.t, M, K) == lib.H3Q_OK
    # the outputs were written (the guards are not intact merely because nothing ran)
    ref = lib.h3q_linear_w8a8(x, qw.t, sw.t, b, want_acc=True)
    assert torch.equal(acc.t, ref["acc"]) and torch.equal(y.t.view(torch.int16),
                                                          ref["y"].view(torch.int16))


@pytest.mark.parametrize("M,K", [(1, 16), (127, 1040), (257, 5376), (32767, 5376), (33, 21504)])
def test_quantize_act_writes_stay_inside_their_buffers(lib, dev, M, K):
    x, _, _ = _operands(M, 1, K, seed=M + K, dev=dev)
    xq = Guarded((M, K), torch.int8, dev)
    xs = Guarded((M,), torch.float32, dev)
    lib.h3q_quantize_act(x, q_out=xq.t, scale_out=xs.t)
    torch.cuda.synchronize()
    assert xq.intact() and xs.intact()


@pytest.mark.parametrize("G,M,N,K", [(3, 257, 131, 5376), (4, 129, 5383, 1040),
                                     (2, 32767, 257, 5376)])
def test_grouped_outputs_stay_inside_their_buffers(lib, dev, G, M, N, K):
    c = synth.make_linear(M, N, K, seed=G * 1000 + M, n_linears=G, outlier_p=0.01,
                          outlier_mul=20.0)
    x = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    qws, sws, bs = [], [], []
    for w, bb in zip(c.w, c.bias_bits):
        q, s = lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
        qws.append(q)
        sws.append(s)
        bs.append(torch.from_numpy(bb.view(np.int16)).view(torch.bfloat16).to(dev))
    ys = [Guarded((M, N), torch.bfloat16, dev) for _ in range(G)]
    xs = Guarded((M,), torch.float32, dev)
    need = lib.h3q_linear_grouped_workspace_bytes(G, M, N, K)
    ws = Guarded((need,), torch.uint8, dev)
    lib.h3q_linear_w8a8_grouped(x, qws, sws, bs, xs=xs.t, ys=[g.t for g in ys], workspace=ws.t)
    torch.cuda.synchronize()
    for i, g in enumerate(ys):
        assert g.intact(), f"output {i}: a guard byte changed"
    assert xs.intact() and ws.intact()


def test_host_pipeline_staging_stays_inside_its_buffers(lib, dev):
    G, M, N, K = 2, 1000, 131, 1040          # chunks of 64, 128, 256, 256, 256, 40 rows
    c = synth.make_linear(M, N, K, seed=77, n_linears=G)
    x_host = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    qws, sws = [], []
    for w in c.w:
        q, s = lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
        qws.append(q)
        sws.append(s)
    x_dev = Guarded((M, K), torch.bfloat16, dev)
    xs = Guarded((M,), torch.float32, dev)
    ys_dev = [Guarded((M, N), torch.bfloat16, dev) for _ in range(G)]
    chunk = 256
    need = lib.h3q_linear_w8a8_grouped_host_workspace_bytes(G, M, N, K, chunk)
    ws = Guarded((need,), torch.uint8, dev)
    out = lib.h3q_linear_w8a8_grouped_host(x_host, qws, sws, None, x_dev=x_dev.t, xs=xs.t,
                                           ys_dev=[g.t for g in ys_dev], chunk_rows=chunk,
                                           first_rows=64, workspace=ws.t)
    torch.cuda.synchronize()
    assert x_dev.intact() and xs.intact() and ws.intact()
    for i, g in enumerate(ys_dev):
        assert g.intact(), f"device output {i}: a guard byte changed"
        assert torch.equal(out["ys"][i].view(torch.int16), g.t.cpu().view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(129, 131, 1040), (1559, 5376, 5376), (7, 1, 16)])
def test_noalloc_writes_stay_inside_their_buffers(lib, dev, M, N, K):
    """The allocation-free entry point writes only its outputs (its scratch is
    internal): guard bands around y, the raw accumulators and the activation
    scales, on ragged shapes up to the built-in scratch's edge (M = 1559 at
    N = K = 5376)."""
    x, w, b = _operands(M, N, K, seed=M + N + K + 5, dev=dev)
    qw, sw = lib.h3q_quantize_weights(w)
    y = Guarded((M, N), torch.bfloat16, dev)
    acc = Guarded((M, N), torch.int32, dev)
    xs = Guarded((M,), torch.float32, dev)
    lib.h3q_linear_w8a8_noalloc(x, qw, sw, b, xs=xs.t, y=y.t, acc_out=acc.t)
    torch.cuda.synchronize()
    assert y.intact() and acc.intact() and xs.intact()
    assert lib.h3q_linear_w8a8_noalloc_status(M, K) == lib.H3Q_OK
    ref = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True)
    assert torch.equal(acc.t, ref["acc"])
    assert torch.equal(y.t.view(torch.int16), ref["y"].view(torch.int16))
