"""GPU parity of the group-wise affine comparison scheme (weight-only; "MLX
implementation and experiment report", Operator tuning: Q8/g64 and Q4/g64).

Bar: codes, steps and offsets bit-exact against the oracle; the Linear's BF16
outputs within one BF16 ulp plus the FP32 accumulation bound K 2^-23
sum_k |x_k w^_k| of the oracle's float64 value (the tensor cores' FP32
summation order is not fixed).
"""
import math

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _bf16_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _check_affine_y(oracle, y_bits, ref, K):
    """|y - v| <= ulp_bf16(v) + K 2^-23 sum|x w^| elementwise."""
    y = oracle.widen_bf16(y_bits).astype(np.float64)
    v = ref["v"]
    av = np.abs(v)
    e = np.floor(np.log2(np.where(av > 0, av, 1.0)))
    ulp = np.where(av >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)
    tol = ulp + K * 2.0 ** -23 * ref["absum"] * 1.0001
    err = np.abs(y - v)
    bad = err > tol
    assert not np.any(bad), (f"{int(bad.sum())} outputs outside the bound; first at "
                             f"{tuple(np.argwhere(bad)[0])}: y {y[bad][0]} v {v[bad][0]}")
    return float(np.max(err / tol))


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_weights_affine_matches_oracle(lib, oracle, dev, dtype, bits):
    rng = np.random.default_rng(80)
    w = (rng.standard_normal((300, 1024)) * 0.02).astype(np.float32)
    w[3, 64:128] = np.float32(0.125)                        # a constant group
    w[7, :64] *= np.float32(1e-36)                          # a tiny-range group
    wt = torch.from_numpy(w).to(dev).to(dtype)
    q, ab = lib.h3q_quantize_weights_affine(wt, bits=bits)
    w_in = wt.float().cpu().numpy()                          # the values the kernel saw
    oq, oa, ob = oracle.quantize_affine(w_in, bits=bits)
    assert int(q.max()) == 2 ** bits - 1 and int(q.min()) == 0
    assert np.array_equal(q.cpu().numpy(), oq)
    got = ab.cpu().numpy()
    assert np.array_equal(got[:, :, 0].view(np.uint32), oa.view(np.uint32))
    assert np.array_equal(got[:, :, 1].view(np.uint32), ob.view(np.uint32))


@pytest.mark.parametrize("bad", [np.inf, np.nan])
def test_quantize_weights_affine_rejects_non_finite(lib, dev, bad):
    w = np.ones((4, 128), np.float32)
    w[2, 70] = bad
    with pytest.raises(lib.H3QError) as e:
        lib.h3q_quantize_weights_affine(torch.from_numpy(w).to(dev))
    assert e.value.status == lib.H3Q_ERR_NONFINITE


@pytest.mark.parametrize("M,N,K,bits", [(1, 1, 64, 8), (7, 3, 128, 8), (129, 264, 192, 8),
                                        (300, 100, 5376, 8), (33, 520, 14336, 8),
                                        (517, 300, 1024, 8), (7, 3, 128, 4), (300, 100, 5376, 4),
                                        (517, 300, 1024, 4)])
def test_linear_affine_parity_ragged(lib, oracle, dev, M, N, K, bits):
    rng = np.random.default_rng(M * 7 + N + K)
    xb = oracle.round_to_bf16(rng.standard_normal((M, K)))
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    bias = oracle.round_to_bf16(rng.standard_normal(N) * 0.1)
    q, ab = lib.h3q_quantize_weights_affine(torch.from_numpy(w).to(dev), bits=bits)
    out = lib.h3q_linear_affine_w8(_bf16_dev(xb, dev), q, ab, _bf16_dev(bias, dev))
    torch.cuda.synchronize()
    assert int(out["status"][0]) == 0
    oq, oa, ob = oracle.quantize_affine(w, bits=bits)
    ref = oracle.linear_affine(xb, oracle.dequant_affine(oq, oa, ob), bias)
    _check_affine_y(oracle, _bits(out["y"]), ref, K)


def test_linear_affine_without_bias_and_zero_rows(lib, oracle, dev):
    rng = np.random.default_rng(81)
    M, N, K = 200, 136, 512
    xb = oracle.round_to_bf16(rng.standard_normal((M, K)))
    xb[5] = 0
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    q, ab = lib.h3q_quantize_weights_affine(torch.from_numpy(w).to(dev))
    out = lib.h3q_linear_affine_w8(_bf16_dev(xb, dev), q, ab)
    torch.cuda.synchronize()
    y = _bits(out["y"])
    assert np.all((y[5] & 0x7FFF) == 0)                      # a zero row gives +-0
    oq, oa, ob = oracle.quantize_affine(w)
    _check_affine_y(oracle, y, oracle.linear_affine(xb, oracle.dequant_affine(oq, oa, ob)), K)


@pytest.mark.parametrize("name", ["image_qkv", "image_down"])
def test_linear_affine_image_workloads_sampled(lib, oracle, dev, name):
    # the H3-Image operator shapes at 4096 tokens: the whole GEMM on the GPU,
    # sampled rows and channels (the first, the last and random ones) checked
    c = synth.WORKLOADS[name]()
    M, K = c.x_bits.shape
    N = c.w[0].shape[0]
    q, ab = lib.h3q_quantize_weights_affine(torch.from_numpy(c.w[0]).to(dev))
    out = lib.h3q_linear_affine_w8(_bf16_dev(c.x_bits, dev), q, ab, _bf16_dev(c.bias_bits[0], dev))
    torch.cuda.synchronize()
    assert int(out["status"][0]) == 0
    rng = np.random.default_rng(82)
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 30)]))
    cols = np.unique(np.concatenate([np.arange(128), [N - 1], rng.integers(0, N, 200)]))
    oq, oa, ob = oracle.quantize_affine(c.w[0][cols])
    ref = oracle.linear_affine(c.x_bits[rows], oracle.dequant_affine(oq, oa, ob),
                               c.bias_bits[0][cols])
    y = out["y"][torch.from_numpy(rows).to(dev)][:, torch.from_numpy(cols).to(dev)]
    _check_affine_y(oracle, _bits(y.contiguous()), ref, K)


@pytest.mark.parametrize("bits,K,jmax", [(8, 1024, 8), (4, 1024, 8), (8, 5376, 4), (4, 5376, 4)])
def test_linear_affine_exact_where_fp32_sums_are_exact(lib, oracle, dev, bits, K, jmax):
    """A tight pin for the comparison scheme's Linear.  The general bound above
    must allow the worst FP32 summation error, since the tensor cores' order is
    not fixed; here the inputs sit on coarse grids that make every product and
    every partial sum exact in FP32, in any order: activations j 2^-3 (|j| <=
    jmax), weights k 2^-6 with every group holding the grid's two ends (so the
    step is exactly 2^-6 and the dequantised weights are the k 2^-6
    themselves), biases on 2^-9.  Then the sums are multiples of 2^-9 below
    2^22 of those units, the bias adds exactly, and each output must be the
    exact value rounded once to BF16, bit for bit."""
    M, N = 300, 264
    rng = np.random.default_rng(90 + bits + K)
    L = 2 ** bits - 1
    kmin, kmax = -(L + 1) // 2, L // 2                      # Q8: -128..127, Q4: -8..7
    kk = rng.integers(kmin, kmax + 1, size=(N, K))
    kk[:, 0::64], kk[:, 1::64] = kmin, kmax
    w = (kk * 2.0 ** -6).astype(np.float32)
    xb = oracle.round_to_bf16(rng.integers(-jmax, jmax + 1, size=(M, K)) * 2.0 ** -3)
    bias = oracle.round_to_bf16(rng.integers(-64, 65, size=N) * 2.0 ** -9)
    q, ab = lib.h3q_quantize_weights_affine(torch.from_numpy(w).to(dev), bits=bits)
    assert bool((ab[:, :, 0] == 2.0 ** -6).all())
    out = lib.h3q_linear_affine_w8(_bf16_dev(xb, dev), q, ab, _bf16_dev(bias, dev))
    torch.cuda.synchronize()
    assert int(out["status"][0]) == 0
    oq, oa, ob = oracle.quantize_affine(w, bits=bits)
    what = oracle.dequant_affine(oq, oa, ob)
    assert np.array_equal(oracle.widen_bf16(what).astype(np.float64), kk * 2.0 ** -6)
    ref = oracle.linear_affine(xb, what, bias)
    assert np.all(ref["absum"] * 2 ** 9 < 2 ** 22)
    got = _bits(out["y"])
    bad = got != ref["y"]
    assert not np.any(bad), (f"{int(bad.sum())} outputs differ from the once-rounded exact "
                             f"value; first at {tuple(np.argwhere(bad)[0])}")
