"""GPU parity of the two ways h3q_linear_w8a8 accumulates a tile.

A tile whose INT8 rows satisfy |a|^2 |w|^2 <= 2^48 (largest squared row norms
of its 256 tokens and 256 channels) keeps all of K in one FP32 accumulator;
any other tile cuts K into chunks of at most 1024.  Both must give the exact
INT32 sum.  These tests drive each path on its own, the boundary case, and a
mix, and check that the split is the one the norms dictate (the expected
split is computed here from the INT8 codes, independently of the library).
"""
import math

import numpy as np
import pytest
import torch

from _parity import check_exact, check_y

pytestmark = pytest.mark.gpu

BOUND = 1 << 48


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _bf16_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def expected_chunked_tiles(qa, qw):
    """128-token x 256-channel tiles that fail the squared-norm bound: per
    256-token block and 256-channel block, max |a|^2 * max |w|^2 > 2^48."""
    M, N = qa.shape[0], qw.shape[0]
    a2 = (qa.astype(np.int64) ** 2).sum(1)
    w2 = (qw.astype(np.int64) ** 2).sum(1)
    mt128 = math.ceil(M / 128)
    count = 0
    for b in range(math.ceil(M / 256)):
        amax = int(a2[256 * b: 256 * b + 256].max())
        for p in range(math.ceil(N / 256)):
            wmax = int(w2[256 * p: 256 * p + 256].max())
            if amax * wmax > BOUND:
                count += min(2, mt128 - 2 * b)
    return count


def _run(lib, oracle, dev, xq, wq, xs, ws, bias):
    acc = oracle.gemm_int32(xq, wq)
    ref = oracle.epilogue_value(acc, xs, ws, bias)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    out = lib.h3q_linear_w8a8(None, t(wq), t(ws), None if bias is None else _bf16_dev(bias, dev),
                              xq=t(xq), xs=t(xs), want_acc=True)
    check_exact(out["acc"].cpu().numpy(), acc, "acc")
    check_y(_bits(out["y"]), ref)
    M, K = xq.shape
    assert lib.h3q_workspace_status(out["workspace"], M, K) == lib.H3Q_OK
    return acc, lib.h3q_linear_chunked_tiles(out["workspace"], M, K)


def _odd_vector_with_square_norm(K, target, seed):
    """Odd-heavy INT8 vector of length K with sum of squares exactly `target`:
    random odd entries while the running sum stays well below the target, the
    rest of it as a sum of four squares, then zeros."""
    rng = np.random.default_rng(seed)
    v = (2 * rng.integers(-63, 64, K) + 1).astype(np.int64)       # odd, in [-125, 127]
    cs = np.cumsum(v * v)
    L = int(np.searchsorted(cs, target - 20000, side="right"))   # keep v[:L]
    rest = target - (int(cs[L - 1]) if L else 0)
    assert 20000 <= rest <= 20000 + 127 * 127 and L + 4 <= K
    two = {}
    for c in range(128):
        for d in range(c + 1):
            two.setdefault(c * c + d * d, (c, d))
    for a in range(127, -1, -1):
        for b in range(a + 1):
            r = rest - a * a - b * b
            if r in two:
                out = np.zeros(K, np.int64)
                out[:L] = v[:L]
                out[L:L + 4] = [a, b, *two[r]]
                assert int((out * out).sum()) == target
                return out
    raise AssertionError("no four-square split")


def test_bound_reached_exactly_takes_the_single_accumulator(lib, oracle, dev):
    # |a|^2 = |w|^2 = 2^24 for every row: the product is exactly 2^48, so every
    # tile keeps all of K in FP32.  Rows are sign flips of one odd-heavy vector
    # v, so acc = sum_k (+-1) v_k^2; the rows with equal signs sum to 2^24
    # through partial sums that climb past 2^23 in odd steps.
    K, M, N = 4096, 293, 200
    v = _odd_vector_with_square_norm(K, 1 << 24, seed=5)
    rng = np.random.default_rng(6)
    sa = np.where(rng.random((M, K)) < 0.5, -1, 1)
    sw = np.where(rng.random((N, K)) < 0.5, -1, 1)
    sa[0] = 1
    sw[0] = 1
    sa[7] = sw[3]
    xq = (sa * v).astype(np.int8)
    wq = (sw * v).astype(np.int8)
    xs = rng.uniform(2.0 ** -9, 2.0 ** -8, M).astype(np.float32)
    ws = rng.uniform(2.0 ** -9, 2.0 ** -8, N).astype(np.float32)
    acc, chunked = _run(lib, oracle, dev, xq, wq, xs, ws, None)
    assert acc[0, 0] == 1 << 24 and acc[7, 3] == 1 << 24
    assert expected_chunked_tiles(xq, wq) == 0
    assert chunked == 0


def test_bound_exceeded_by_one_row_takes_the_chunked_path(lib, oracle, dev):
    # the same rows, with one token row of the first 256-token block raised
    # above the bound: that block (two 128-token tiles) goes to the chunked
    # path, the ragged second block stays on the single accumulator
    K, M, N = 4096, 293, 200
    v = _odd_vector_with_square_norm(K, 1 << 24, seed=5)
    xq = np.tile(v, (M, 1)).astype(np.int8)
    wq = np.tile(v, (N, 1)).astype(np.int8)
    j = int(np.argmax(np.abs(v) < 120))
    xq[100, j] += 3 if v[j] >= 0 else -3
    rng = np.random.default_rng(8)
    xs = rng.uniform(0.5, 1.0, M).astype(np.float32) * 2.0 ** -10
    ws = rng.uniform(0.5, 1.0, N).astype(np.float32) * 2.0 ** -10
    bias = (rng.integers(0, 2 ** 15, N) & 0x7F7F).astype(np.uint16)
    acc, chunked = _run(lib, oracle, dev, xq, wq, xs, ws, bias)
    assert expected_chunked_tiles(xq, wq) == 2
    assert chunked == 2
    assert acc[0, 0] == 1 << 24 and acc[100, 0] > 1 << 24


def test_mixed_tiles(lib, oracle, dev):
    # per-block amplitudes put some tiles above the bound and some below:
    # token blocks of 256 with |q| up to {20, 127, 40, 127, 90}, channel
    # blocks of 256 with |q| up to {30, 127, 60}; the last of each is ragged
    K, M, N = 8192, 1100, 700
    rng = np.random.default_rng(9)
    amp_m = np.repeat([20, 127, 40, 127, 90], 256)[:M]
    amp_n = np.repeat([30, 127, 60], 256)[:N]
    xq = np.round(rng.uniform(-1, 1, (M, K)) * amp_m[:, None]).astype(np.int8)
    wq = np.round(rng.uniform(-1, 1, (N, K)) * amp_n[:, None]).astype(np.int8)
    xs = rng.uniform(2.0 ** -12, 2.0 ** -11, M).astype(np.float32)
    ws = rng.uniform(2.0 ** -12, 2.0 ** -11, N).astype(np.float32)
    bias = (rng.integers(0, 2 ** 15, N) & 0xBF7F).astype(np.uint16)
    exp = expected_chunked_tiles(xq, wq)
    total = math.ceil(M / 128) * math.ceil(N / 256)
    assert 0 < exp < total
    _, chunked = _run(lib, oracle, dev, xq, wq, xs, ws, bias)
    assert chunked == exp


def test_every_tile_chunked(lib, oracle, dev):
    # constant +-127 rows: |a|^2 |w|^2 = (127^2 K)^2 > 2^48 everywhere
    K, M, N = 2048, 300, 520
    rng = np.random.default_rng(10)
    xq = np.where(rng.random((M, K)) < 0.5, -127, 127).astype(np.int8)
    wq = np.where(rng.random((N, K)) < 0.5, -127, 127).astype(np.int8)
    xs = np.full(M, 2.0 ** -7, np.float32)
    ws = np.full(N, 2.0 ** -7, np.float32)
    _, chunked = _run(lib, oracle, dev, xq, wq, xs, ws, None)
    assert chunked == math.ceil(M / 128) * math.ceil(N / 256)
