"""The 300-Linear sweep configuration (M = 75647 packed tokens; per DiT block
Q, K, V, O [5376 -> 5376], FC1 [5376 -> 21504], FC2 [21504 -> 5376]) at full
size, on the first and the last block, against the oracle on sampled token
rows (the first 128, the last 128 and 128 seeded ones, all N columns).  The
tensors come from the sweep's seeded device generator; the oracle gets the
same bytes copied to the host.  The INT8 weights and scales are compared
whole."""
import numpy as np
import pytest
import torch

import synth
from _parity import check_exact, check_y

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def sweep_inputs(dev):
    return {K: synth.sweep_x(K, dev) for K in (synth.H3_WIDTH, synth.H3_MLP_WIDTH)}


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _sample_rows(M, seed, n_rand=128):
    rng = np.random.default_rng(seed)
    rand = rng.choice(M, size=n_rand, replace=False)
    return np.unique(np.concatenate([np.arange(128), np.arange(M - 128, M), rand]))


@pytest.mark.parametrize("block", [0, 49])
def test_sweep_block_sampled(lib, oracle, dev, sweep_inputs, block):
    M = synth.SWEEP_M
    rows = _sample_rows(M, 500 + block)
    rt = torch.from_numpy(rows).to(dev)
    for j, (name, N, K) in enumerate(synth.SWEEP_LINEARS):
        w, b = synth.sweep_weight(block, j, dev)
        qw, sw = lib.h3q_quantize_weights(w)
        qw_ref, sw_ref = oracle.quantize_weights(w.cpu().numpy())
        check_exact(qw.cpu().numpy(), qw_ref, f"{name} q_w")
        check_exact(sw.cpu().numpy(), sw_ref, f"{name} s_w")
        del w
        x = sweep_inputs[K]
        out = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True, want_xq=True)
        ref = oracle.linear(_bits(x[rt]), qw_ref, sw_ref, _bits(b))
        check_exact(out["xq"][rt].cpu().numpy(), ref["qa"], f"{name} q_a")
        check_exact(out["xs"][rt].cpu().numpy(), ref["sa"], f"{name} s_a")
        check_exact(out["acc"][rt].cpu().numpy(), ref["acc"], f"{name} acc")
        check_y(_bits(out["y"][rt]), ref["v"], f"{name} y")
        assert lib.h3q_workspace_status(out["workspace"], M, K) == lib.H3Q_OK
        del out
        torch.cuda.empty_cache()


def test_sweep_block0_fc2_every_row_against_the_legacy_exact_kernel(lib, dev, sweep_inputs):
    """Block 0's FC2 (75647 x 5376 x 21504): every output against the legacy
    mma.sync INT8 kernel on the same INT8 operands (exact by construction and
    oracle-checked on its own), so every tile's accumulation path is checked."""
    j = 5
    name, N, K = synth.SWEEP_LINEARS[j]
    M = synth.SWEEP_M
    w, b = synth.sweep_weight(0, j, dev)
    qw, sw = lib.h3q_quantize_weights(w)
    del w
    out = lib.h3q_linear_w8a8(sweep_inputs[K], qw, sw, b, want_acc=True, want_xq=True)
    ws = out.pop("workspace")
    ckpt = lib.h3q_linear_checkpointed_tiles(ws, M, K)
    del ws
    torch.cuda.empty_cache()
    leg = lib.h3q_linear_w8a8_mma_sync(out["xq"], out["xs"], qw, sw, b, want_acc=True)
    torch.cuda.synchronize()
    bad = int((out["acc"] != leg["acc"]).sum())
    assert bad == 0, f"{name}: {bad} INT32 accumulators differ from the legacy exact kernel"
    assert torch.equal(out["y"].view(torch.int16), leg["y"].view(torch.int16))
    assert ckpt >= 0
