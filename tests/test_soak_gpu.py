"""A seeded random-shape soak of h3q_linear_w8a8 against the legacy mma.sync
INT8 kernel (exact by construction, itself checked against the oracle).

Shapes (ragged M and N, K any multiple of 16 up to 22384) and input
distributions (Gaussian with outliers, uniform, signs only so that every code
is +-127, SiLU-like) are drawn so that tiles take every accumulation path: one
FP32 accumulator, checkpoints, and the chunked kernel.  Each call's INT32
accumulators and BF16 outputs must equal the legacy kernel's bit for bit, with
a clean status word.  The loop runs for a fixed time budget.
"""
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BUDGET_S = 15.0


def _inputs(kind, M, N, K, g, dev):
    if kind == 0:      # Gaussian with 0.5 % outliers x30
        x = torch.randn((M, K), generator=g, device=dev)
        x = torch.where(torch.rand((M, K), generator=g, device=dev) < 0.005, x * 30, x)
        w = torch.randn((N, K), generator=g, device=dev) * 0.02
    elif kind == 1:    # uniform: large codes everywhere
        x = torch.rand((M, K), generator=g, device=dev) * 2 - 1
        w = torch.rand((N, K), generator=g, device=dev) * 2 - 1
    elif kind == 2:    # signs only: every code +-127
        x = torch.sign(torch.randn((M, K), generator=g, device=dev)) + 0.0
        w = torch.sign(torch.randn((N, K), generator=g, device=dev)) + 0.0
    else:              # SiLU of a normal draw: non-negative skew
        z = torch.randn((M, K), generator=g, device=dev)
        x = z * torch.sigmoid(z)
        w = torch.randn((N, K), generator=g, device=dev) * 0.01
    return x.to(torch.bfloat16), w


def test_random_shapes_match_the_legacy_exact_kernel(lib):
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(20261203)
    t0 = time.time()
    calls = ckpt = chunked = 0
    while time.time() - t0 < BUDGET_S:
        M = int(rng.choice([1, 7, 64, 129, 255, 256, 257, 511, 1000, 2049, 4096]))
        N = int(rng.choice([1, 8, 131, 256, 257, 512, 1000, 2048]))
        K = int(16 * rng.integers(1, 1400))
        kind = int(rng.integers(0, 4))
        g = torch.Generator(device=dev)
        g.manual_seed(int(rng.integers(1 << 31)))
        x, w = _inputs(kind, M, N, K, g, dev)
        qw, sw = lib.h3q_quantize_weights(w)
        b = ((torch.randn((N,), generator=g, device=dev) * 0.1).to(torch.bfloat16)
             if rng.integers(0, 2) else None)
        out = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True, want_xq=True)
        leg = lib.h3q_linear_w8a8_mma_sync(out["xq"], out["xs"], qw, sw, b, want_acc=True)
        torch.cuda.synchronize()
        what = f"M={M} N={N} K={K} inputs={kind} bias={b is not None}"
        assert lib.h3q_workspace_status(out["workspace"], M, K) == lib.H3Q_OK, what
        assert torch.equal(out["acc"], leg["acc"]), f"{what}: INT32 accumulators differ"
        assert torch.equal(out["y"].view(torch.int16), leg["y"].view(torch.int16)), \
            f"{what}: BF16 outputs differ"
        ckpt += lib.h3q_linear_checkpointed_tiles(out["workspace"], M, K) > 0
        chunked += lib.h3q_linear_chunked_tiles(out["workspace"], M, K) > 0
        calls += 1
    # the budget covers many calls, and both the checkpointed and the chunked path
    assert calls > 100 and ckpt > 0 and chunked > 0, (calls, ckpt, chunked)


def test_random_grouped_calls_match_separate_calls(lib):
    """The grouped launch on random shapes: G = 1..4 Linears sharing X (their
    tiles interleaved in one launch, with per-Linear fallback lists), each
    output equal bit for bit to that Linear's own single call, and the
    activation scales equal too.  Seeded; a fixed time budget."""
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(20261204)
    t0 = time.time()
    calls = 0
    while time.time() - t0 < BUDGET_S:
        G = int(rng.integers(1, 5))
        M = int(rng.choice([1, 33, 256, 257, 700, 2049]))
        N = int(rng.choice([8, 130, 257, 512, 1000]))
        K = int(16 * rng.integers(1, 1400))
        kind = int(rng.integers(0, 4))
        g = torch.Generator(device=dev)
        g.manual_seed(int(rng.integers(1 << 31)))
        x, _ = _inputs(kind, M, 1, K, g, dev)
        qws, sws, bs = [], [], []
        for i in range(G):
            _, w = _inputs(kind, 1, N, K, g, dev)
            q, s = lib.h3q_quantize_weights(w)
            qws.append(q)
            sws.append(s)
            bs.append((torch.randn((N,), generator=g, device=dev) * 0.1).to(torch.bfloat16)
                      if rng.integers(0, 2) else None)
        out = lib.h3q_linear_w8a8_grouped(x, qws, sws, bs)
        for i in range(G):
            one = lib.h3q_linear_w8a8(x, qws[i], sws[i], bs[i])
            torch.cuda.synchronize()
            what = f"G={G} Linear {i} M={M} N={N} K={K} inputs={kind}"
            assert torch.equal(one["xs"], out["xs"]), f"{what}: activation scales differ"
            assert torch.equal(one["y"].view(torch.int16), out["ys"][i].view(torch.int16)), \
                f"{what}: outputs differ from the single call"
        calls += 1
    assert calls > 30, calls
