"""GPU parity of h3q_linear_w8a8_grouped: G Linears that share their input in
one GEMM launch give, bit for bit, what one h3q_linear_w8a8 call per Linear
gives (and so match the oracle within one BF16 ulp), in every mode: BF16
input, pre-quantised input, and reuse of the coded activations."""
import math

import numpy as np
import pytest
import torch

import synth
from _parity import check_y

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _bf16_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,N,K,G", [(300, 264, 5376, 3), (129, 128, 1040, 2), (513, 520, 2048, 4),
                                     (64, 256, 5376, 1)])
def test_grouped_matches_separate_calls_and_oracle(lib, oracle, dev, M, N, K, G):
    c = synth.make_linear(M, N, K, seed=M + G, n_linears=G, outlier_p=0.005, outlier_mul=30)
    x = _bf16_dev(c.x_bits, dev)
    q = [lib.h3q_quantize_weights(torch.from_numpy(w).to(dev)) for w in c.w]
    b = [_bf16_dev(bb, dev) for bb in c.bias_bits]
    if G >= 2:
        b[1] = None                                  # one Linear without a bias
    grp = lib.h3q_linear_w8a8_grouped(x, [w for w, _ in q], [s for _, s in q], b)
    for g in range(G):
        one = lib.h3q_linear_w8a8(x, q[g][0], q[g][1], b[g])
        assert _same(grp["ys"][g], one["y"]), f"Linear {g} differs from its own call"
        ref = oracle.linear(c.x_bits, *oracle.quantize_weights(c.w[g]),
                            None if b[g] is None else c.bias_bits[g])
        check_y(_bits(grp["ys"][g]), ref["v"])
    assert lib.h3q_workspace_status(grp["workspace"], M, K) == lib.H3Q_OK


def test_grouped_prequantised_and_reuse_modes(lib, dev):
    M, N, K, G = 200, 136, 5376, 3
    c = synth.make_linear(M, N, K, seed=61, n_linears=G)
    x = _bf16_dev(c.x_bits, dev)
    q = [lib.h3q_quantize_weights(torch.from_numpy(w).to(dev)) for w in c.w]
    wq, ws = [w for w, _ in q], [s for _, s in q]
    b = [_bf16_dev(bb, dev) for bb in c.bias_bits]
    first = lib.h3q_linear_w8a8_grouped(x, wq, ws, b)
    xq, xs = lib.h3q_quantize_act(x)
    pre = lib.h3q_linear_w8a8_grouped(None, wq, ws, b, xq=xq, xs=xs)
    again = lib.h3q_linear_w8a8_grouped(None, wq, ws, b, xs=first["xs"],
                                        workspace=first["workspace"])
    for g in range(G):
        assert _same(pre["ys"][g], first["ys"][g])
        assert _same(again["ys"][g], first["ys"][g])


def test_grouped_with_chunked_tiles(lib, oracle, dev):
    # Linear 0's weights keep every tile on the single accumulator; Linear 1's
    # send the token block of full-magnitude one-sign rows to the chunked
    # path and keep the uniform-code block on one accumulator by checkpoints
    K, M, N = 8192, 600, 300
    rng = np.random.default_rng(62)
    amp_m = np.repeat([20, 127, 40], 256)[:M]
    xq = np.round(rng.uniform(-1, 1, (M, K)) * amp_m[:, None]).astype(np.int8)
    xq[:128] = (np.where(rng.random(128) < 0.5, -127, 127)[:, None] *
                np.ones(K, np.int64)).astype(np.int8)
    wq0 = np.round(rng.uniform(-1, 1, (N, K)) * 10).astype(np.int8)
    wq1 = np.round(rng.uniform(-1, 1, (N, K)) * 127).astype(np.int8)
    xs = rng.uniform(2.0 ** -12, 2.0 ** -11, M).astype(np.float32)
    ws = [rng.uniform(2.0 ** -12, 2.0 ** -11, N).astype(np.float32) for _ in range(2)]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    grp = lib.h3q_linear_w8a8_grouped(None, [t(wq0), t(wq1)], [t(w) for w in ws], None,
                                      xq=t(xq), xs=t(xs))
    counts = []
    for g, wq in enumerate((wq0, wq1)):
        one = lib.h3q_linear_w8a8(None, t(wq), t(ws[g]), None, xq=t(xq), xs=t(xs))
        assert _same(grp["ys"][g], one["y"])
        counts.append((lib.h3q_linear_chunked_tiles(one["workspace"], M, K),
                       lib.h3q_linear_checkpointed_tiles(one["workspace"], M, K)))
        ref = oracle.epilogue_value(oracle.gemm_int32(xq, wq), xs, ws[g], None)
        check_y(_bits(grp["ys"][g]), ref)
    assert counts[0] == (0, 0) and counts[1][0] > 0 and counts[1][1] > 0
    assert lib.h3q_linear_chunked_tiles(grp["workspace"], M, K) == sum(c[0] for c in counts)
    assert lib.h3q_linear_checkpointed_tiles(grp["workspace"], M, K) == sum(c[1] for c in counts)


@pytest.mark.slow
def test_grouped_attn_workload_matches_separate_calls(lib, dev):
    c = synth.attn()
    x = _bf16_dev(c.x_bits, dev)
    q = [lib.h3q_quantize_weights(torch.from_numpy(w).to(dev)) for w in c.w]
    b = [_bf16_dev(bb, dev) for bb in c.bias_bits]
    grp = lib.h3q_linear_w8a8_grouped(x, [w for w, _ in q], [s for _, s in q], b)
    for g in range(4):
        one = lib.h3q_linear_w8a8(x, q[g][0], q[g][1], b[g])
        assert _same(grp["ys"][g], one["y"])


def test_grouped_call_replays_from_a_cuda_graph(lib, dev):
    # a call that does not synchronise enqueues everything on the caller's
    # stream (the memset and the programmatic-dependent launches), so it can be
    # captured in a CUDA graph; replays give the eager call's bits
    M, N, K, G = 300, 264, 5376, 3
    c = synth.make_linear(M, N, K, seed=93, n_linears=G, outlier_p=0.005, outlier_mul=30)
    x = _bf16_dev(c.x_bits, dev)
    q = [lib.h3q_quantize_weights(torch.from_numpy(w).to(dev)) for w in c.w]
    wq, ws = [w for w, _ in q], [s for _, s in q]
    b = [_bf16_dev(bb, dev) for bb in c.bias_bits]
    ref = lib.h3q_linear_w8a8_grouped(x, wq, ws, b)
    ys = [torch.empty_like(y) for y in ref["ys"]]
    xs = torch.empty_like(ref["xs"])
    work = torch.empty_like(ref["workspace"])
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        lib.h3q_linear_w8a8_grouped(x, wq, ws, b, xs=xs, ys=ys, workspace=work, stream=side)
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            lib.h3q_linear_w8a8_grouped(x, wq, ws, b, xs=xs, ys=ys, workspace=work, stream=side)
    for rep in range(2):
        for y in ys:
            y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for g in range(G):
            assert _same(ys[g], ref["ys"][g]), (rep, g)
        assert lib.h3q_workspace_status(work, M, K) == lib.H3Q_OK
