"""GPU parity of h3q_linear_w8a8_grouped_host: the grouped Linear from and to
page-locked host memory, pipelined in row chunks.  Whatever the chunk plan,
its host outputs equal, bit for bit, the device outputs of one
h3q_linear_w8a8_grouped call on the same operands (A2 is per token and each
output element depends on its own token row only), and match the oracle
within one BF16 ulp."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _parity import check_exact, check_y

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _same(a, b):
    return torch.equal(a.view(torch.int16).cpu(), b.view(torch.int16).cpu())


def _operands(lib, c, dev, G, drop_bias):
    q = [lib.h3q_quantize_weights(torch.from_numpy(w).to(dev)) for w in c.w]
    b = [_bf16(bb).to(dev) for bb in c.bias_bits]
    if drop_bias and G >= 2:
        b[1] = None                                  # one Linear without a bias
    return [w for w, _ in q], [s for _, s in q], b


# (M, N, K, G, chunk_rows, first_rows): a ramp 64, 128, 256 then steady chunks
# and a ragged last one; many 16-row chunks; one chunk larger than M; the
# default first chunk.
@pytest.mark.parametrize("M,N,K,G,chunk,first", [(1000, 264, 1040, 3, 256, 64),
                                                 (77, 136, 5376, 2, 16, 16),
                                                 (300, 128, 512, 4, 4096, 0),
                                                 (129, 520, 2048, 1, 32, 0)])
def test_host_pipeline_matches_grouped_call_and_oracle(lib, oracle, dev, M, N, K, G, chunk,
                                                       first):
    c = synth.make_linear(M, N, K, seed=M + G + chunk, n_linears=G, outlier_p=0.005,
                          outlier_mul=30)
    wq, ws, b = _operands(lib, c, dev, G, drop_bias=True)
    x_host = _bf16(c.x_bits).pin_memory()
    out = lib.h3q_linear_w8a8_grouped_host(x_host, wq, ws, b, chunk_rows=chunk, first_rows=first)
    ref = lib.h3q_linear_w8a8_grouped(x_host.to(dev), wq, ws, b)
    torch.cuda.synchronize()
    assert torch.equal(out["xs"].cpu(), ref["xs"].cpu())
    assert _same(out["x_dev"], x_host)
    for g in range(G):
        assert _same(out["ys"][g], ref["ys"][g]), f"Linear {g}: host output differs"
        assert _same(out["ys_dev"][g], ref["ys"][g])
        want = oracle.linear(c.x_bits, *oracle.quantize_weights(c.w[g]),
                             None if b[g] is None else c.bias_bits[g])
        check_exact(out["xs"].cpu().numpy(), want["sa"], "s_a")
        check_y(_bits(out["ys"][g]), want["v"])


def test_host_pipeline_on_one_stream(lib, dev):
    # uploads, calls and downloads all on the current stream, into separately
    # allocated outputs (one download per output and chunk): serial, and the
    # same result as three streams with one [G, M, N] buffer (2D downloads)
    M, N, K, G = 500, 200, 1040, 2
    c = synth.make_linear(M, N, K, seed=71, n_linears=G)
    wq, ws, b = _operands(lib, c, dev, G, drop_bias=False)
    x_host = _bf16(c.x_bits).pin_memory()
    s = torch.cuda.current_stream(dev)
    sep_host = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(G)]
    sep_dev = [torch.empty((M + 1, N), dtype=torch.bfloat16, device=dev)[:M] for _ in range(G)]
    one = lib.h3q_linear_w8a8_grouped_host(x_host, wq, ws, b, ys_host=sep_host, ys_dev=sep_dev,
                                           chunk_rows=128, h2d_stream=s, d2h_stream=s)
    three = lib.h3q_linear_w8a8_grouped_host(x_host, wq, ws, b, chunk_rows=128)
    for g in range(G):
        assert _same(one["ys"][g], three["ys"][g])


def test_host_pipeline_rejects_pageable_host_memory(lib, dev):
    M, N, K = 64, 64, 64
    f = lib.load().h3q_linear_w8a8_grouped_host
    x_pageable = torch.zeros((M, K), dtype=torch.bfloat16)
    y_pinned = torch.zeros((M, N), dtype=torch.bfloat16).pin_memory()
    y_pageable = torch.zeros((M, N), dtype=torch.bfloat16)
    x_pinned = torch.zeros((M, K), dtype=torch.bfloat16).pin_memory()
    wq = torch.zeros((N, K), dtype=torch.int8, device=dev)
    ws = torch.ones((N,), dtype=torch.float32, device=dev)
    x_dev = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    xs = torch.empty((M,), dtype=torch.float32, device=dev)
    y_dev = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    nbytes = lib.h3q_linear_w8a8_grouped_host_workspace_bytes(1, M, N, K, 32)
    work = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
    one = lambda t: (ctypes.c_void_p * 1)(t.data_ptr())
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    call = lambda xh, yh: f(vp(xh), 1, one(wq), one(ws), None, M, N, K, one(yh), vp(x_dev),
                            vp(xs), one(y_dev), 32, 0, vp(work), nbytes, s, s, s)
    assert call(x_pageable, y_pinned) == lib.H3Q_ERR_INVALID_ARG
    assert call(x_pinned, y_pageable) == lib.H3Q_ERR_INVALID_ARG
    assert call(x_pinned, y_pinned) == lib.H3Q_OK
    assert torch.count_nonzero(y_pinned.view(torch.int16)) == 0     # zero weights, no bias


@pytest.mark.slow
def test_host_pipeline_attn_workload(lib, oracle, dev):
    # the attention step through host memory, in the bench's chunking:
    # every output equals the device call's; sampled rows (the first rows of
    # every chunk, the tail and random rows) against the oracle
    c = synth.attn()
    G = len(c.w)
    wq, ws, b = _operands(lib, c, dev, G, drop_bias=False)
    x_host = _bf16(c.x_bits).pin_memory()
    out = lib.h3q_linear_w8a8_grouped_host(x_host, wq, ws, b, chunk_rows=1024)
    ref = lib.h3q_linear_w8a8_grouped(x_host.to(dev), wq, ws, b)
    torch.cuda.synchronize()
    for g in range(G):
        assert _same(out["ys"][g], ref["ys"][g]), f"Linear {g}: host output differs"
    rng = np.random.default_rng(111)
    starts = [0, 256, 768] + list(range(1792, c.M, 1024))
    rows = np.unique(np.concatenate([np.array(starts), np.array(starts[1:]) - 1,
                                     np.arange(c.M - 8, c.M), rng.choice(c.M, 48, replace=False)]))
    for g in range(G):
        want = oracle.linear(c.x_bits[rows], *oracle.quantize_weights(c.w[g]), c.bias_bits[g])
        check_y(_bits(out["ys"][g][torch.from_numpy(rows)]), want["v"])


def test_host_pipeline_equally_spaced_outputs(lib, oracle, dev):
    # the G outputs as one [G, M, N] buffer on each side: a chunk's downloads
    # go as one 2D copy; the results are those of the grouped device call
    M, N, K, G = 700, 264, 1040, 3
    c = synth.make_linear(M, N, K, seed=97, n_linears=G, outlier_p=0.005, outlier_mul=30)
    wq, ws, b = _operands(lib, c, dev, G, drop_bias=True)
    x_host = _bf16(c.x_bits).pin_memory()
    yh = torch.zeros((G, M, N), dtype=torch.bfloat16).pin_memory()
    yd = torch.empty((G, M, N), dtype=torch.bfloat16, device=dev)
    out = lib.h3q_linear_w8a8_grouped_host(x_host, wq, ws, b, ys_host=[yh[g] for g in range(G)],
                                           ys_dev=[yd[g] for g in range(G)], chunk_rows=256,
                                           first_rows=48)
    ref = lib.h3q_linear_w8a8_grouped(x_host.to(dev), wq, ws, b)
    torch.cuda.synchronize()
    for g in range(G):
        assert _same(yh[g], ref["ys"][g]), f"Linear {g}: host output differs"
        assert _same(yd[g], ref["ys"][g])
        want = oracle.linear(c.x_bits, *oracle.quantize_weights(c.w[g]),
                             None if b[g] is None else c.bias_bits[g])
        check_y(_bits(yh[g]), want["v"])
    assert out["ys"][0].data_ptr() == yh[0].data_ptr()


def test_prepared_host_call_repeats_on_new_inputs(lib, oracle, dev):
    """GroupedHostCall checks and marshals once; each call reads the current
    contents of x_host and gives what the one-shot function gives on it."""
    M, N, K, G = 700, 264, 1040, 3
    c1 = synth.make_linear(M, N, K, seed=91, n_linears=G, outlier_p=0.005, outlier_mul=30)
    c2 = synth.make_linear(M, N, K, seed=92, n_linears=G, outlier_p=0.005, outlier_mul=30)
    wq, ws, b = _operands(lib, c1, dev, G, drop_bias=True)
    x_host = _bf16(c1.x_bits).pin_memory()
    call = lib.GroupedHostCall(x_host, wq, ws, b, chunk_rows=256, first_rows=64)
    for c in (c1, c2, c1):
        x_host.copy_(_bf16(c.x_bits))
        ys = [y.clone() for y in call()]
        ref = lib.h3q_linear_w8a8_grouped_host(x_host, wq, ws, b, chunk_rows=256, first_rows=64)
        for g in range(G):
            assert _same(ys[g], ref["ys"][g]), f"Linear {g}: prepared call differs"
    want = oracle.linear(c1.x_bits, *oracle.quantize_weights(c1.w[0]), c1.bias_bits[0])
    check_y(_bits(ys[0]), want["v"])


def test_prepared_host_call_checks_its_arguments(lib, dev):
    M, N, K = 64, 64, 64
    wq = [torch.zeros((N, K), dtype=torch.int8, device=dev)]
    ws = [torch.ones((N,), dtype=torch.float32, device=dev)]
    with pytest.raises(TypeError):
        lib.GroupedHostCall(torch.zeros((M, K), dtype=torch.bfloat16), wq, ws)   # not pinned
    with pytest.raises(TypeError):
        lib.GroupedHostCall(torch.zeros((M, K), dtype=torch.float32).pin_memory(), wq, ws)
    with pytest.raises(ValueError):
        lib.GroupedHostCall(torch.zeros((M, K + 16), dtype=torch.bfloat16).pin_memory(), wq, ws)
