"""GPU parity of the ways h3q_linear_w8a8 accumulates a tile.

A tile whose INT8 rows satisfy |a|^2 |w|^2 <= 2^48 (largest squared row norms
of its 256 tokens and 256 channels) keeps all of K in one FP32 accumulator.
A tile that fails that test can still keep one accumulator by checkpoints:
K is cut into four norm segments, runs of segments are bounded by
Cauchy-Schwarz on the per-segment norms, and between runs the kernel reads
the accumulator's largest magnitude and proves that the next run stays
within 2^24.  Any other tile, or a checkpointed one whose proof fails, is
recomputed with K cut into chunks of at most 1024.  All must give the exact
INT32 sum.  These tests drive each path, the boundary case, and mixes, and
check that the split is the one the rules dictate: `tile_paths` below
computes it from the INT8 codes with numpy, independently of the library.
"""
import math

import numpy as np
import pytest
import torch

from _parity import check_exact, check_y

pytestmark = pytest.mark.gpu

BOUND = 1 << 48
EXACT = 1 << 24                  # FP32 holds every integer up to this
RUN_LIMIT = EXACT - (1 << 21)    # a planned run's bound leaves room for the start value
SEGS = 4


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _bf16_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def segment_len(K):
    """Norm segment length: a quarter of the 128-element super-stages, rounded up."""
    return math.ceil(math.ceil(K / 128) / SEGS) * 128


def tile_paths(qa, qw):
    """(chunked 128 x 256 tiles, checkpointed 256 x 256 tiles) under the rules:
    a 256-token x 256-channel tile is exact on one accumulator if
    max|a|^2 * 128^2 K or max|a|^2 * max|w|^2 is <= 2^48; otherwise runs of
    norm segments grow while (sum of the tile's per-segment token maxima) x
    (sum of its channel maxima) <= RUN_LIMIT^2, a checkpoint starting each new
    run, and a segment that alone exceeds it (or the first) sends the tile to
    the chunked path; at each checkpoint the exact partial sums so far give
    obs = max |S| over the tile, and the tile falls back to the chunked path
    unless (2^24 - obs)^2 >= (the next run's norm sums product)."""
    M, K = qa.shape
    N = qw.shape[0]
    sl, nss = segment_len(K), math.ceil(K / 128)
    a2 = qa.astype(np.int64) ** 2
    w2 = qw.astype(np.int64) ** 2
    a_full, w_full = a2.sum(1), w2.sum(1)
    a_seg = np.stack([a2[:, s * sl:(s + 1) * sl].sum(1) for s in range(SEGS)], 1)
    w_seg = np.stack([w2[:, s * sl:(s + 1) * sl].sum(1) for s in range(SEGS)], 1)
    qa64, qw64 = qa.astype(np.float64), qw.astype(np.float64)
    mt128 = math.ceil(M / 128)
    chunked = ckpt = 0
    for b in range(math.ceil(M / 256)):
        rows = slice(256 * b, 256 * b + 256)
        A = int(a_full[rows].max())
        As = [int(v) for v in a_seg[rows].max(0)]
        for p in range(math.ceil(N / 256)):
            cols = slice(256 * p, 256 * p + 256)
            if A * 128 * 128 * K <= BOUND or A * int(w_full[cols].max()) <= BOUND:
                continue
            Ws = [int(v) for v in w_seg[cols].max(0)]
            ra = rw = 0
            plan, to_chunked = [], False
            for i in range(SEGS):
                if i * (sl // 128) >= nss:
                    break
                na, nw = ra + As[i], rw + Ws[i]
                if na * nw <= RUN_LIMIT ** 2:
                    ra, rw = na, nw
                    continue
                if i == 0 or As[i] * Ws[i] > RUN_LIMIT ** 2:
                    to_chunked = True
                    break
                plan.append(i)
                ra, rw = As[i], Ws[i]
            if to_chunked:
                chunked += min(2, mt128 - 2 * b)
                continue
            if not plan:
                continue
            ckpt += 1
            failed = False
            for j, s in enumerate(plan):
                S = qa64[rows, :s * sl] @ qw64[cols, :s * sl].T     # exact: < 2^53
                obs = int(np.abs(S).max())
                end = plan[j + 1] if j + 1 < len(plan) else SEGS
                ar, wr = sum(As[s:end]), sum(Ws[s:end])
                if obs > EXACT or (EXACT - obs) ** 2 < ar * wr:
                    failed = True
            if failed:
                chunked += min(2, mt128 - 2 * b)
    return chunked, ckpt


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
    got = (lib.h3q_linear_chunked_tiles(out["workspace"], M, K),
           lib.h3q_linear_checkpointed_tiles(out["workspace"], M, K))
    assert got == tile_paths(xq, wq)
    return acc, got


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
    acc, paths = _run(lib, oracle, dev, xq, wq, xs, ws, None)
    assert acc[0, 0] == 1 << 24 and acc[7, 3] == 1 << 24
    assert paths == (0, 0)


def test_bound_exceeded_by_one_row_takes_the_chunked_path(lib, oracle, dev):
    # the same rows, with one token row of the first 256-token block raised
    # above the bound: that block's tile takes checkpoints, but its partial
    # sums (all of one sign) do reach past 2^24, so the proof fails and the
    # chunked path recomputes it (two 128-token tiles); the ragged second
    # block stays on the single accumulator
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
    acc, paths = _run(lib, oracle, dev, xq, wq, xs, ws, bias)
    assert paths == (2, 1)
    assert acc[0, 0] == 1 << 24 and acc[100, 0] > 1 << 24


def test_mixed_tiles(lib, oracle, dev):
    # per-block amplitudes put some tiles within the whole-K bound, some
    # within reach of checkpoints and some beyond: token blocks of 256 with
    # |q| up to {20, 127, 40, 127, 90}, the second of them made of rows of
    # one sign and full magnitude; channel blocks of 256 with |q| up to
    # {30, 127, 60}; the last of each is ragged
    K, M, N = 8192, 1100, 700
    rng = np.random.default_rng(9)
    amp_m = np.repeat([20, 127, 40, 127, 90], 256)[:M]
    amp_n = np.repeat([30, 127, 60], 256)[:N]
    xq = np.round(rng.uniform(-1, 1, (M, K)) * amp_m[:, None]).astype(np.int8)
    wq = np.round(rng.uniform(-1, 1, (N, K)) * amp_n[:, None]).astype(np.int8)
    xq[256:512] = (np.where(rng.random(256) < 0.5, -127, 127)[:, None] *
                   np.ones(K, np.int64)).astype(np.int8)
    xs = rng.uniform(2.0 ** -12, 2.0 ** -11, M).astype(np.float32)
    ws = rng.uniform(2.0 ** -12, 2.0 ** -11, N).astype(np.float32)
    bias = (rng.integers(0, 2 ** 15, N) & 0xBF7F).astype(np.uint16)
    chunked, ckpt = tile_paths(xq, wq)
    total = math.ceil(M / 128) * math.ceil(N / 256)
    assert 0 < chunked < total and ckpt > 0
    _run(lib, oracle, dev, xq, wq, xs, ws, bias)


def test_every_tile_chunked(lib, oracle, dev):
    # constant +-127 rows with K = 8192: each quarter of K alone has
    # |a|^2 |w|^2 = (127^2 2048)^2 above the run limit, so no tile can take
    # checkpoints and every tile goes straight to the chunked path
    K, M, N = 8192, 300, 520
    rng = np.random.default_rng(10)
    xq = np.where(rng.random((M, K)) < 0.5, -127, 127).astype(np.int8)
    wq = np.where(rng.random((N, K)) < 0.5, -127, 127).astype(np.int8)
    xs = np.full(M, 2.0 ** -7, np.float32)
    ws = np.full(N, 2.0 ** -7, np.float32)
    _, paths = _run(lib, oracle, dev, xq, wq, xs, ws, None)
    assert paths == (math.ceil(M / 128) * math.ceil(N / 256), 0)


def test_uniform_codes_take_checkpoints(lib, oracle, dev):
    # codes uniform in [-127, 127] with K = 4096: |a|^2 |w|^2 is about 1.7 x
    # 2^48, so no tile passes the whole-K test, but half of K stays within
    # the run limit and the random-walk partial sums stay far below 2^24:
    # every tile keeps one accumulator with one checkpoint
    K, M, N = 4096, 600, 520
    rng = np.random.default_rng(11)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    xs = rng.uniform(2.0 ** -12, 2.0 ** -11, M).astype(np.float32)
    ws = rng.uniform(2.0 ** -12, 2.0 ** -11, N).astype(np.float32)
    bias = (rng.integers(0, 2 ** 15, N) & 0xBF7F).astype(np.uint16)
    _, paths = _run(lib, oracle, dev, xq, wq, xs, ws, bias)
    assert paths == (0, math.ceil(M / 256) * math.ceil(N / 256))


def test_failed_checkpoints_fall_back(lib, oracle, dev):
    # rows of one sign and magnitude (+-127 times a per-row sign) with
    # K = 2048: every quarter of K passes the run limit, so every tile takes
    # checkpoints, but the partial sums grow linearly to 127^2 K > 2^24, the
    # second checkpoint's proof fails, and the chunked path recomputes every
    # tile
    K, M, N = 2048, 300, 520
    rng = np.random.default_rng(12)
    xq = (np.where(rng.random(M) < 0.5, -127, 127)[:, None] * np.ones(K, np.int64)).astype(np.int8)
    wq = (np.where(rng.random(N) < 0.5, -127, 127)[:, None] * np.ones(K, np.int64)).astype(np.int8)
    xs = np.full(M, 2.0 ** -9, np.float32)
    ws = np.full(N, 2.0 ** -9, np.float32)
    acc, paths = _run(lib, oracle, dev, xq, wq, xs, ws, None)
    assert paths == (math.ceil(M / 128) * math.ceil(N / 256),
                     math.ceil(M / 256) * math.ceil(N / 256))
    assert abs(int(acc[0, 0])) == 127 * 127 * K


def _workspace_norms(ws, M, K):
    """The activation norm maxima a Linear call leaves in its workspace: per
    256-token block the largest sum of q^2 of a row, then per block and norm
    segment (the workspace starts with the FP16-coded activations, rows of
    ceil(K / 64) * 64 elements, each part 256-byte aligned)."""
    up = lambda b: (b + 255) // 256 * 256
    mt = math.ceil(M / 256)
    off = up(M * math.ceil(K / 64) * 64 * 2)
    w = ws.cpu().numpy()[off:off + 4 * mt * (1 + SEGS)].view(np.uint32)
    return w[:mt], w[mt:].reshape(mt, SEGS)


@pytest.mark.parametrize("M,K", [(700, 5376), (300, 14336), (37, 2064)])
def test_norm_maxima_from_bf16_input(lib, oracle, dev, M, K):
    # the quantiser inside the call records, besides the codes and scales, the
    # per-block and per-segment maxima of the rows' sums of q^2 that decide the
    # tile paths; compare them with the oracle's codes
    rng = np.random.default_rng(13 + K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[rng.random((M, K)) < 0.003] *= 25.0
    x[5] = 0.0                                    # an all-zero row
    xb = oracle.round_to_bf16(x)
    w = (rng.standard_normal((40, K)) * 0.02).astype(np.float32)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
    out = lib.h3q_linear_w8a8(_bf16_dev(xb, dev), qw, sw, None)
    torch.cuda.synchronize()
    qa, _ = oracle.quantize_act(xb)
    a2 = qa.astype(np.int64) ** 2
    sl = segment_len(K)
    full, seg = _workspace_norms(out["workspace"], M, K)
    for b in range(math.ceil(M / 256)):
        rows = slice(256 * b, 256 * b + 256)
        assert int(full[b]) == int(a2[rows].sum(1).max())
        for s in range(SEGS):
            assert int(seg[b, s]) == int(a2[rows, s * sl:(s + 1) * sl].sum(1).max())


def test_tile_paths_and_outputs_are_deterministic(lib, oracle, dev):
    # R9: every output is bitwise identical run to run, whichever way each tile
    # went.  Here tiles take all three ways (one accumulator, checkpoints, the
    # chunked kernel): ten calls must agree bit for bit, in their path counts
    # too.
    K, M, N = 4096, 900, 520
    rng = np.random.default_rng(14)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)              # checkpoints hold
    xq[:256] = np.round(rng.uniform(-1, 1, (256, K)) * 20).astype(np.int8)   # one accumulator
    xq[512:768] = (np.where(rng.random(256) < 0.5, -127, 127)[:, None] *
                   np.ones(K, np.int64)).astype(np.int8)              # chunked against wq[:256]
    wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    wq[:256] = np.where(rng.random((256, K)) < 0.5, -127, 127)
    xs = rng.uniform(2.0 ** -12, 2.0 ** -11, M).astype(np.float32)
    ws = rng.uniform(2.0 ** -12, 2.0 ** -11, N).astype(np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    paths = tile_paths(xq, wq)
    assert paths[0] > 0 and paths[1] > 0
    first = None
    for _ in range(10):
        out = lib.h3q_linear_w8a8(None, t(wq), t(ws), None, xq=t(xq), xs=t(xs), want_acc=True)
        got = (lib.h3q_linear_chunked_tiles(out["workspace"], M, K),
               lib.h3q_linear_checkpointed_tiles(out["workspace"], M, K))
        assert got == paths
        y = out["y"].view(torch.int16).clone()
        if first is None:
            first = (y, out["acc"].clone())
            check_exact(out["acc"].cpu().numpy(), oracle.gemm_int32(xq, wq), "acc")
        else:
            assert torch.equal(y, first[0]) and torch.equal(out["acc"], first[1])


@pytest.mark.parametrize("K", [1152, 1408])
def test_checkpoints_with_uneven_segments(lib, oracle, dev, K):
    # K = 1152: nine super-stages in segments of 3, 3, 3 and an empty fourth;
    # K = 1408: eleven in 3, 3, 3, 2.  Random +-127 codes fail the whole-K test
    # (|a|^2 |w|^2 up to 2 x 2^48) but hold with one checkpoint before the third
    # segment; the planner must skip the empty segment and size the last run
    # from the segments that exist
    M, N = 300, 520
    rng = np.random.default_rng(15 + K)
    xq = np.where(rng.random((M, K)) < 0.5, -127, 127).astype(np.int8)
    wq = np.where(rng.random((N, K)) < 0.5, -127, 127).astype(np.int8)
    xs = np.full(M, 2.0 ** -9, np.float32)
    ws = np.full(N, 2.0 ** -9, np.float32)
    _, paths = _run(lib, oracle, dev, xq, wq, xs, ws, None)
    assert paths == (0, math.ceil(M / 256) * math.ceil(N / 256))


def test_mixed_paths_match_the_legacy_exact_path(lib, oracle, dev):
    # 9 token blocks x 9 channel-block pairs = 81 cluster tiles on every path
    # at once.  Token block 8's activations are all +-127.  Against them,
    # channel pair 4's +-127 weights fail even the per-segment test (the
    # chunked kernel takes the tile), pair 5's single-outlier rows pass the
    # whole-K test (one accumulator), and the Gaussian rows of pairs 6-8 pass
    # only per segment (checkpoints); the other token blocks mix the first two.
    # Every output and accumulator must equal the legacy mma.sync path's,
    # which is exact INT32 by construction, bit for bit.
    M, N, K = 2304, 2176, 8192
    rng = np.random.default_rng(95)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[2048:] = np.where(rng.random((M - 2048, K)) < 0.5, -1.0, 1.0)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[1024:1280] = np.where(rng.random((256, K)) < 0.5, -0.02, 0.02)
    w[1280:1536] = rng.standard_normal((256, K)).astype(np.float32) * 1e-4
    w[1280:1536, 7] = 0.5
    xb = oracle.round_to_bf16(x)
    b = oracle.round_to_bf16(rng.standard_normal(N) * 0.1)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
    xt, bt = _bf16_dev(xb, dev), _bf16_dev(b, dev)
    out = lib.h3q_linear_w8a8(xt, qw, sw, bt, want_acc=True, want_xq=True)
    chunked = lib.h3q_linear_chunked_tiles(out["workspace"], M, K)
    ckpt = lib.h3q_linear_checkpointed_tiles(out["workspace"], M, K)
    legacy = lib.h3q_linear_w8a8_mma_sync(out["xq"], out["xs"], qw, sw, bt, want_acc=True)
    torch.cuda.synchronize()
    assert torch.equal(out["acc"], legacy["acc"])
    assert torch.equal(out["y"].view(torch.int16), legacy["y"].view(torch.int16))
    assert chunked >= 2, chunked                    # pair 4 of block 8: two 128-token tiles
    assert ckpt >= 3, ckpt                          # pairs 6-8 of block 8, at least
    rows = np.unique(np.concatenate([np.arange(2040, 2056), np.arange(M - 8, M),
                                     rng.integers(0, M, 16)]))
    ref = oracle.linear(xb[rows], *oracle.quantize_weights(w), b)
    rt = torch.from_numpy(rows).to(dev)
    check_exact(out["acc"][rt].cpu().numpy(), ref["acc"], "acc")
    check_y(_bits(out["y"][rt]), ref["v"])
