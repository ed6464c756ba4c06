"""GPU parity: the CUDA path through the C-ABI against the CPU oracle.

Bar: INT8 activations and weights, FP32 scales and INT32 accumulators
bit-exact; BF16 outputs within one BF16 ulp of the oracle's float64 epilogue
value.  Inputs come from the seeded generators in ``synth`` and are the same
bytes on both sides.
"""
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


def _bf16_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _special_rows(K, rng):
    """Rows that exercise the quantiser's edge cases, as BF16 bits."""
    rows = [np.zeros(K, np.uint16),                                   # all zero -> s = 1
            np.full(K, 0x8000, np.uint16),                            # all -0.0
            np.full(K, 0x3F40, np.uint16),                            # constant 0.75 -> 127
            np.full(K, 0xBD00, np.uint16)]                            # constant -1/32 -> -127
    sub = np.zeros(K, np.uint16); sub[::3] = 0x0001; sub[1::3] = 0x8003   # subnormals
    rows.append(sub)
    # power-of-two scale (absmax 127 * 2^-3) with exact ties k + 0.5
    tie = np.array([(k % 60) - 30 + 0.5 for k in range(K)], np.float32) / 8
    tie[0] = 127.0 / 8
    rows.append(synth.to_bf16_bits(tie))
    big = rng.standard_normal(K).astype(np.float32); big[K // 2] = 3.0e38
    rows.append(synth.to_bf16_bits(big))                              # huge outlier
    return np.stack(rows)


def _act(M, K, seed, special=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    m = rng.random((M, K)) < 0.01
    x[m] *= 25
    bits = synth.to_bf16_bits(x)
    if special:
        sp = _special_rows(K, rng)
        n = min(len(sp), M)
        bits[-n:] = sp[:n]
    return bits


@pytest.mark.parametrize("M,K", [(1, 16), (7, 48), (129, 5376), (64, 6144), (33, 6160),
                                 (300, 21504), (9, 133136)])
def test_quantize_act_bit_exact(lib, oracle, dev, M, K):
    xb = _act(M, K, seed=M * 7 + K)
    q, s = lib.h3q_quantize_act(_bf16_dev(xb, dev))
    oq, os_ = oracle.quantize_act(xb)
    check_exact(q.cpu().numpy(), oq, "q_a")
    check_exact(s.cpu().numpy(), os_, "s_a")


@pytest.mark.parametrize("N,K", [(1, 16), (100, 80), (256, 5376), (37, 21504)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_quantize_weights_bit_exact(lib, oracle, dev, N, K, dtype):
    rng = np.random.default_rng(N + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[0, :] = 0.0                                   # zero row -> scale 1
    if N > 2:
        w[1, :] = np.float32(1e-44)                 # subnormal row
        w[2, 3] = np.float32(2.0 ** -149)           # smallest subnormal in a row
    if dtype == "bf16":
        wb = synth.to_bf16_bits(w)
        wt = _bf16_dev(wb, dev)
        oq, os_ = oracle.quantize_weights(wb)
    else:
        wt = torch.from_numpy(w).to(dev)
        oq, os_ = oracle.quantize_weights(w)
    q, s = lib.h3q_quantize_weights(wt)
    check_exact(q.cpu().numpy(), oq, "q_w")
    check_exact(s.cpu().numpy(), os_, "s_w")


def test_weight_underflow_scale(lib, oracle, dev):
    w = np.zeros((2, 32), np.float32)
    w[0, 5] = np.float32(2.0 ** -149) * 3        # absmax / 127 underflows to 0
    w[1, 7] = -np.float32(2.0 ** -149) * 63
    q, s = lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
    oq, os_ = oracle.quantize_weights(w)
    check_exact(q.cpu().numpy(), oq, "q_w")
    check_exact(s.cpu().numpy(), os_, "s_w")
    assert float(s[0]) == 2.0 ** -149


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_quantize_weights_rejects_non_finite(lib, dev, bad):
    w = np.ones((8, 64), np.float32)
    w[5, 9] = bad
    with pytest.raises(lib.H3QError) as e:
        lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
    assert e.value.status == lib.H3Q_ERR_NONFINITE


def _linear_check(lib, oracle, dev, xb, w, bias_bits, rows=None, **kw):
    wt = torch.from_numpy(w).to(dev)
    qw, sw = lib.h3q_quantize_weights(wt)
    oq, osw = oracle.quantize_weights(w)
    check_exact(qw.cpu().numpy(), oq, "q_w")
    check_exact(sw.cpu().numpy(), osw, "s_w")
    bias = None if bias_bits is None else _bf16_dev(bias_bits, dev)
    out = lib.h3q_linear_w8a8(_bf16_dev(xb, dev), qw, sw, bias, want_acc=True, want_xq=True, **kw)
    torch.cuda.synchronize()
    if rows is None:
        rows = np.arange(xb.shape[0])
    rt = torch.from_numpy(rows).to(dev)
    ref = oracle.linear(xb[rows], oq, osw, bias_bits)
    check_exact(out["xq"][rt].cpu().numpy(), ref["qa"], "q_a")
    check_exact(out["xs"][rt].cpu().numpy(), ref["sa"], "s_a")
    check_exact(out["acc"][rt].cpu().numpy(), ref["acc"], "acc")
    stats = check_y(_bits(out["y"][rt]), ref["v"])
    return out, stats


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (7, 3, 48), (129, 264, 80), (300, 100, 5376),
                                   (33, 8, 21504), (130, 257, 64), (5, 131, 1040)])
def test_linear_parity_ragged(lib, oracle, dev, M, N, K):
    rng = np.random.default_rng(M * 1000 + N)
    xb = _act(M, K, seed=M + N + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    bias = synth.to_bf16_bits((rng.standard_normal(N) * 0.1).astype(np.float32))
    _linear_check(lib, oracle, dev, xb, w, bias)


def test_linear_tiny_workload(lib, oracle, dev):
    c = synth.tiny()
    _, stats = _linear_check(lib, oracle, dev, c.x_bits, c.w[0], c.bias_bits[0])
    assert stats["max_ulp"] <= 1.0


def test_linear_without_bias_and_output_selection(lib, oracle, dev):
    c = synth.make_linear(70, 136, 5376, seed=21)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
    x = _bf16_dev(c.x_bits, dev)
    ref = oracle.linear(c.x_bits, *oracle.quantize_weights(c.w[0]), None)
    out = lib.h3q_linear_w8a8(x, qw, sw, None, want_y=True, want_acc=False)
    check_y(_bits(out["y"]), ref["v"])
    out = lib.h3q_linear_w8a8(x, qw, sw, None, want_y=False, want_acc=True)
    check_exact(out["acc"].cpu().numpy(), ref["acc"], "acc")


def test_linear_prequantised_input(lib, oracle, dev):
    c = synth.make_linear(96, 200, 5376, seed=22)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
    xq, xs = lib.h3q_quantize_act(_bf16_dev(c.x_bits, dev))
    bias = _bf16_dev(c.bias_bits[0], dev)
    out = lib.h3q_linear_w8a8(None, qw, sw, bias, xq=xq, xs=xs, want_acc=True)
    ref = oracle.linear(c.x_bits, *oracle.quantize_weights(c.w[0]), c.bias_bits[0])
    check_exact(out["acc"].cpu().numpy(), ref["acc"], "acc")
    check_y(_bits(out["y"]), ref["v"])


@pytest.mark.parametrize("K", [5376, 21504, 133136])
def test_linear_extreme_accumulators(lib, oracle, dev, K):
    # constant rows quantise to +-127, so acc = +-127^2 K: the largest
    # accumulators the shape allows (K = 133136 is the largest legal K)
    M, N = 3, 4
    xb = np.zeros((M, K), np.uint16)
    xb[0] = 0x3F80; xb[1] = 0xBF80                  # +-1.0
    xb[2, ::2] = 0x3F80; xb[2, 1::2] = 0xBF80       # alternating
    w = np.ones((N, K), np.float32)
    w[1] *= -1
    w[2, : K // 2] = -1
    w[3, ::3] = 0.5
    out, _ = _linear_check(lib, oracle, dev, xb, w, None)
    assert int(out["acc"][0, 0]) == 127 * 127 * K
    assert int(out["acc"][1, 0]) == -127 * 127 * K


def test_linear_partial_sums_cross_2_pow_24(lib, oracle, dev):
    # running sums exceed 2^24 and come back: exact INT32 required
    K, M, N = 5376, 4, 8
    xb = np.full((M, K), 0x3F80, np.uint16)
    xb[1, K // 3:] = 0xBF80
    xb[2, ::7] = 0x3F00
    w = np.ones((N, K), np.float32)
    w[0, K // 2:] = -1
    w[1, -1] = 0.5
    w[2, 1::2] = -1
    w[3, : 1030] = -1
    out, _ = _linear_check(lib, oracle, dev, xb, w, None)


def test_deterministic(lib, dev):
    c = synth.make_linear(257, 384, 5376, seed=31)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
    x = _bf16_dev(c.x_bits, dev)
    b = _bf16_dev(c.bias_bits[0], dev)
    o1 = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True)
    o2 = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True)
    assert torch.equal(o1["y"].view(torch.int16), o2["y"].view(torch.int16))
    assert torch.equal(o1["acc"], o2["acc"])


def test_misaligned_device_pointer_rejected(lib, dev):
    M, K, N = 4, 64, 8
    flat = torch.zeros(M * K + 1, dtype=torch.bfloat16, device=dev)
    x = flat[1:].view(M, K)                       # contiguous, 2 bytes off alignment
    with pytest.raises(lib.H3QError) as e:
        lib.h3q_quantize_act(x)
    assert e.value.status == lib.H3Q_ERR_MISALIGNED


# --- the named workloads at full size, sampled rows ---------------------------------

def _sample_rows(M, seed, n_rand=128):
    rng = np.random.default_rng(seed)
    head = np.arange(min(128, M))
    tail = np.arange(max(0, M - 128), M)
    rand = rng.choice(M, size=min(n_rand, M), replace=False)
    return np.unique(np.concatenate([head, tail, rand]))


@pytest.mark.slow
def test_attn_workload_sampled(lib, oracle, dev):
    c = synth.attn()
    rows = _sample_rows(c.M, 101)
    for i, nm in enumerate(c.linear_names):
        _linear_check(lib, oracle, dev, c.x_bits, c.w[i], c.bias_bits[i], rows=rows)


@pytest.mark.slow
def test_fc1_workload_sampled(lib, oracle, dev):
    c = synth.fc1()
    _linear_check(lib, oracle, dev, c.x_bits, c.w[0], c.bias_bits[0], rows=_sample_rows(c.M, 102))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["image_qkv", "image_gate_up", "image_down"])
def test_image_operator_shapes_sampled(lib, oracle, dev, name):
    # the H3-Image operator shapes at 4096 tokens (secondary workload)
    c = synth.WORKLOADS[name]()
    _linear_check(lib, oracle, dev, c.x_bits, c.w[0], c.bias_bits[0],
                  rows=_sample_rows(c.M, 105 + len(name)))


@pytest.fixture(scope="module")
def fc2_case():
    return synth.fc2()


@pytest.mark.slow
def test_fc2_workload_sampled(lib, oracle, dev, fc2_case):
    c = fc2_case
    _linear_check(lib, oracle, dev, c.x_bits, c.w[0], c.bias_bits[0], rows=_sample_rows(c.M, 103))


@pytest.mark.slow
def test_fc2_every_row_against_the_legacy_exact_kernel(lib, dev, fc2_case):
    """All 32768 x 5376 outputs of fc2 against the legacy mma.sync INT8 kernel
    on the same INT8 operands.  That kernel is exact by construction (INT32
    accumulation in the instruction) and is itself checked against the oracle
    (test_legacy_mma_sync_entry_point), so every 256-token tile's path --
    single accumulator, checkpoints, or the chunked kernel -- is checked here,
    not only the sampled rows.  y must match bit for bit as well: the output
    depends on (acc, s_a, s_w, bias) alone."""
    c = fc2_case
    x = _bf16_dev(c.x_bits, dev)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
    b = _bf16_dev(c.bias_bits[0], dev)
    out = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True, want_xq=True)
    del x
    ckpt = lib.h3q_linear_checkpointed_tiles(out["workspace"], c.M, c.K)
    leg = lib.h3q_linear_w8a8_mma_sync(out["xq"], out["xs"], qw, sw, b, want_acc=True)
    torch.cuda.synchronize()
    bad = int((out["acc"] != leg["acc"]).sum())
    assert bad == 0, f"{bad} INT32 accumulators differ from the legacy exact kernel"
    assert torch.equal(out["y"].view(torch.int16), leg["y"].view(torch.int16))
    # the workload does exercise the checkpointed path (about half its tiles)
    assert ckpt > 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["fc1", "image_qkv", "image_down"])
def test_workload_every_row_against_the_legacy_exact_kernel(lib, dev, name):
    """The same every-row check as fc2's on three more full-size workloads:
    fc1 (ragged M = 32767, 21504 channels), the H3-Image fused QKV and
    image_down, where every tile keeps one accumulator only by way of a
    checkpoint.  INT32 accumulators and BF16 outputs must equal the legacy
    exact kernel's bit for bit."""
    c = synth.WORKLOADS[name]()
    x = _bf16_dev(c.x_bits, dev)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
    b = _bf16_dev(c.bias_bits[0], dev)
    out = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True, want_xq=True)
    del x
    ckpt = lib.h3q_linear_checkpointed_tiles(out["workspace"], c.M, c.K)
    leg = lib.h3q_linear_w8a8_mma_sync(out["xq"], out["xs"], qw, sw, b, want_acc=True)
    torch.cuda.synchronize()
    bad = int((out["acc"] != leg["acc"]).sum())
    assert bad == 0, f"{name}: {bad} INT32 accumulators differ from the legacy exact kernel"
    assert torch.equal(out["y"].view(torch.int16), leg["y"].view(torch.int16))
    if name == "image_down":
        assert ckpt > 0           # the checkpointed path is the one under test here


@pytest.mark.slow
def test_attn_grouped_step_every_row_against_the_legacy_exact_kernel(lib, dev):
    """The headline step itself: one grouped call over Q, K, V and O of the
    attention workload (8192 x 5376 x 5376 each).  Every output of the four
    Linears must equal, bit for bit, the legacy mma.sync INT8 kernel's on the
    same INT8 operands (that kernel is exact by construction and checked
    against the oracle, and y depends on (acc, s_a, s_w, bias) alone).  The
    activation codes come from h3q_quantize_act, whose scales must equal the
    grouped call's."""
    c = synth.attn()
    x = _bf16_dev(c.x_bits, dev)
    qws, sws, bs = [], [], []
    for w, bb in zip(c.w, c.bias_bits):
        q, s = lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
        qws.append(q)
        sws.append(s)
        bs.append(_bf16_dev(bb, dev))
    out = lib.h3q_linear_w8a8_grouped(x, qws, sws, bs)
    xq, xs = lib.h3q_quantize_act(x)
    del x
    torch.cuda.synchronize()
    assert torch.equal(out["xs"], xs), "the grouped call's activation scales differ from A2's"
    for g in range(4):
        leg = lib.h3q_linear_w8a8_mma_sync(xq, xs, qws[g], sws[g], bs[g])
        torch.cuda.synchronize()
        bad = int((out["ys"][g].view(torch.int16) != leg["y"].view(torch.int16)).sum())
        assert bad == 0, f"Linear {'QKVO'[g]}: {bad} outputs differ from the legacy exact kernel"


def test_epilogue_deep_cancellation(lib, oracle, dev):
    # Row 0's bias is -BF16(acc * s_a * s_w), so v there is the small residual
    # left after cancellation; an FP32 evaluation that rounds the product first
    # can miss it by many BF16 ulps.  Pre-quantised inputs with full-mantissa
    # scales make the products carry all 48 bits.
    rng = np.random.default_rng(77)
    M, N, K = 64, 8192, 64
    xq = rng.integers(-127, 128, (M, K), dtype=np.int8)
    wq = rng.integers(-127, 128, (N, K), dtype=np.int8)
    xs = (rng.uniform(0.5, 1.0, M) * 2.0 ** -6).astype(np.float32)
    ws = (rng.uniform(0.5, 1.0, N) * 2.0 ** -7).astype(np.float32)
    acc = oracle.gemm_int32(xq, wq)
    p0 = oracle.epilogue_value(acc[:1], xs[:1], ws, None)[0]
    bias = oracle.round_to_bf16(-p0)
    ref = oracle.epilogue_value(acc, xs, ws, bias)
    t = lambda a: torch.from_numpy(a).to(dev)
    out = lib.h3q_linear_w8a8(None, t(wq), t(ws), _bf16_dev(bias, dev), xq=t(xq), xs=t(xs),
                              want_acc=True)
    check_exact(out["acc"].cpu().numpy(), acc, "acc")
    check_y(_bits(out["y"]), ref)
    # the construction reaches cancellations deeper than FP32 rounding of the product
    assert np.sum(np.abs(ref[0]) < 2.0 ** -16 * np.abs(p0)) >= 10


def test_epilogue_extreme_scales(lib, oracle, dev):
    # scale products that overflow or underflow FP32 while the exact result
    # is a finite (or zero) BF16 value, and true overflow to +-inf
    M, N, K = 4, 8, 16
    xq = np.full((M, K), 100, np.int8); xq[1] = -100; xq[3, ::2] = 0
    wq = np.full((N, K), 90, np.int8); wq[:, 1] = -7
    xs = np.array([2.0 ** 100, 2.0 ** 100, 2.0 ** -100, 3.0e-20], np.float32)
    ws = np.array([2.0 ** -110, 2.0 ** 20, 2.0 ** -60, 2.0 ** -40, 1.0, 2.0 ** 60,
                   2.0 ** -126, 5.0e-30], np.float32)
    acc = oracle.gemm_int32(xq, wq)
    bias = synth.to_bf16_bits(np.linspace(-1, 1, N).astype(np.float32))
    ref = oracle.epilogue_value(acc, xs, ws, bias)
    t = lambda a: torch.from_numpy(a).to(dev)
    out = lib.h3q_linear_w8a8(None, t(wq), t(ws), _bf16_dev(bias, dev), xq=t(xq), xs=t(xs),
                              want_acc=True)
    check_exact(out["acc"].cpu().numpy(), acc, "acc")
    check_y(_bits(out["y"]), ref)


def test_linear_reuse_mode_shares_the_quantised_input(lib, oracle, dev):
    # Q quantises X into the workspace; K and V reuse it (x = xq = NULL)
    c = synth.make_linear(200, 136, 5376, seed=23, n_linears=3, outlier_p=0.005, outlier_mul=30)
    x = _bf16_dev(c.x_bits, dev)
    outs, refs = [], []
    ws_buf = None
    xs = None
    for i in range(3):
        qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[i]).to(dev))
        b = _bf16_dev(c.bias_bits[i], dev)
        if i == 0:
            o = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True)
            ws_buf, xs = o["workspace"], o["xs"]
        else:
            o = lib.h3q_linear_w8a8(None, qw, sw, b, xs=xs, workspace=ws_buf, want_acc=True)
        outs.append(o)
        refs.append(oracle.linear(c.x_bits, *oracle.quantize_weights(c.w[i]), c.bias_bits[i]))
    assert lib.h3q_workspace_status(ws_buf, 200, 5376) == lib.H3Q_OK
    for o, r in zip(outs, refs):
        check_exact(o["acc"].cpu().numpy(), r["acc"], "acc")
        check_y(_bits(o["y"]), r["v"])


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (130, 257, 64), (300, 100, 5376), (64, 256, 21504)])
def test_legacy_mma_sync_entry_point(lib, oracle, dev, M, N, K):
    c = synth.make_linear(M, N, K, seed=M + N, outlier_p=0.01, outlier_mul=20)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
    xq, xs = lib.h3q_quantize_act(_bf16_dev(c.x_bits, dev))
    out = lib.h3q_linear_w8a8_mma_sync(xq, xs, qw, sw, _bf16_dev(c.bias_bits[0], dev),
                                       want_acc=True)
    ref = oracle.linear(c.x_bits, *oracle.quantize_weights(c.w[0]), c.bias_bits[0])
    check_exact(out["acc"].cpu().numpy(), ref["acc"], "acc")
    check_y(_bits(out["y"]), ref["v"])


def test_workspace_status_after_a_normal_call(lib, dev):
    c = synth.make_linear(300, 400, 2048, seed=41)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
    o = lib.h3q_linear_w8a8(_bf16_dev(c.x_bits, dev), qw, sw, None)
    assert lib.h3q_workspace_status(o["workspace"], 300, 2048) == lib.H3Q_OK


def test_output_bits_depend_on_the_operands_only(lib, dev):
    # A4 forms y from (acc, s_a, s_w, bias) by the same FP32 operations on
    # every path, so the bits cannot depend on how a row was computed: with or
    # without the raw accumulators, in one call or in row chunks that end
    # inside a 32-token block, on the hot kernel or the legacy mma.sync one.
    # Half a million outputs make near-ties of the BF16 rounding certain, where
    # two different FP32 evaluations would disagree.
    M, N, K = 1000, 520, 5376
    c = synth.make_linear(M, N, K, seed=91, outlier_p=0.005, outlier_mul=30)
    x = _bf16_dev(c.x_bits, dev)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
    b = _bf16_dev(c.bias_bits[0], dev)
    full = lib.h3q_linear_w8a8(x, qw, sw, b, want_xq=True)
    with_acc = lib.h3q_linear_w8a8(x, qw, sw, b, want_acc=True)
    parts = [lib.h3q_linear_w8a8(x[r0:r1].contiguous(), qw, sw, b)["y"]
             for r0, r1 in ((0, 100), (100, 333), (333, 1000))]
    legacy = lib.h3q_linear_w8a8_mma_sync(full["xq"], full["xs"], qw, sw, b)
    torch.cuda.synchronize()
    ref = full["y"].view(torch.int16)
    assert torch.equal(with_acc["y"].view(torch.int16), ref)
    assert torch.equal(torch.cat(parts).view(torch.int16), ref)
    assert torch.equal(legacy["y"].view(torch.int16), ref)


def test_quantize_act_waits_for_the_kernel_that_writes_x(lib, oracle, dev):
    """h3q_quantize_act is launched with programmatic dependent launch: its
    blocks may start while the previous kernel on the stream is finishing, and
    must wait for it before reading X.  Here a kernel rewrites X right before
    each call (alternating between two inputs; both are enqueued behind a
    GPU-side sleep, so the quantiser's launch is processed while the copy runs);
    every call's codes and scales must be those of the X just written."""
    M, K = 8192, 5376
    srcs = [_act(M, K, seed=s, special=False) for s in (11, 12)]
    refs = [oracle.quantize_act(b) for b in srcs]
    src_dev = [_bf16_dev(b, dev) for b in srcs]
    x = torch.empty_like(src_dev[0])
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    s = torch.empty((M,), dtype=torch.float32, device=dev)
    rows = torch.arange(0, M, 97, device=dev)
    for i in range(6):
        torch.cuda._sleep(1_000_000)             # keep the GPU busy while both are enqueued
        x.copy_(src_dev[i % 2])                  # the producer kernel
        lib.h3q_quantize_act(x, q, s)
        got_q = q[rows].cpu().numpy()
        got_s = s.cpu().numpy()
        rq, rs = refs[i % 2]
        check_exact(got_q, rq[rows.cpu().numpy()], f"q_a after write {i}")
        check_exact(got_s, rs, f"s_a after write {i}")
