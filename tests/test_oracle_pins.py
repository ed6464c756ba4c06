"""Pins for the CPU oracle: each check compares the oracle with something other
than itself -- exact rational arithmetic, hand-derived closed forms, invariants
of the definition, brute force in Python integers, or a library routine on a
special case -- so that a dropped term, a wrong sign, a transposed operand or a
wrong rounding rule in the oracle fails at least one of them.

Rules pinned (sources by page title and section):
  "feat(mps): support MiniMax-H3 INT8 inference on Apple M5" (LightX2V #1672):
     Validation -- INT8 weights, finite positive FP32 per-channel scales, CPU
     INT32 references, unquantised tensors preserved byte-for-byte;
     Summary by CodeRabbit -- activation quantiser with masked tails.
  "MLX implementation and experiment report" (MiniMax-H3-Image-mlx RESULTS.md):
     What the default preserves -- bias added before the one output rounding.
"""
import hashlib
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --- exact IEEE binary32 rounding, written in rationals for the brute force ------

def _fp32_rn(x: Fraction) -> Fraction:
    """Round a rational to the nearest IEEE binary32 value, ties to even."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * quantum


def _rne_int(x: Fraction) -> int:
    fl = x.numerator // x.denominator
    rem = x - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def _brute_quantize_row(xs):
    xs = [Fraction(float(v)) for v in xs]
    a = max(abs(v) for v in xs)
    if a == 0:
        return [0] * len(xs), Fraction(1)
    s = _fp32_rn(a / 127)
    if s == 0:
        s = Fraction(2) ** -149
    q = [max(-127, min(127, _rne_int(_fp32_rn(v / s)))) for v in xs]
    return q, s


def test_fp32_rn_helper_agrees_with_hardware_on_samples():
    # the helper itself checked against float32 arithmetic on plain cases
    rng = np.random.default_rng(7)
    for _ in range(200):
        a, b = rng.standard_normal(2).astype(np.float32)
        exact = Fraction(float(a)) / Fraction(float(b))
        assert _fp32_rn(exact) == Fraction(float(np.float32(a) / np.float32(b)))


# --- quantiser ------------------------------------------------------------------

def _rows_for_brute_force():
    rng = np.random.default_rng(11)
    rows = [rng.standard_normal(40).astype(np.float32) for _ in range(4)]
    rows.append((rng.standard_normal(40) * 0.02).astype(np.float32))           # weight-like
    r = rng.standard_normal(40).astype(np.float32); r[3] *= 30; rows.append(r)  # outlier
    rows.append(np.float32(1e-38) * rng.standard_normal(40).astype(np.float32))  # subnormal-ish
    rows.append(np.array([np.float32(2.0 ** -149) * k for k in range(-20, 20)], np.float32))
    # ties built on a power-of-two scale (absmax 127 * 2^-2)
    rows.append(np.array([31.75] + [(k + 0.5) / 4 for k in range(-20, 19)], np.float32))
    return rows


def test_quantize_matches_exact_rational_brute_force(oracle):
    rows = _rows_for_brute_force()
    for r in rows:
        q, s = oracle.quantize_rows(r[None, :])
        bq, bs = _brute_quantize_row(r)
        assert Fraction(float(s[0])) == bs
        assert q[0].tolist() == bq


def test_quantize_golden_power_of_two_rows(oracle):
    for row in _load("quant_pow2_rows.json")["rows"]:
        x = np.array(row["x"], np.float32)[None, :]
        q, s = oracle.quantize_rows(x)
        assert q[0].tolist() == row["q"]
        if row["scale"] is not None:
            assert float(s[0]) == row["scale"]


def _dists():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    yield "normal", x
    m = rng.random((64, 512)) < 0.01
    y = x.copy(); y[m] *= 20
    yield "outliers", y
    z = rng.standard_normal((64, 512))
    yield "silu", (z / (1 + np.exp(-z))).astype(np.float32)
    yield "weights", (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    yield "tiny", (rng.standard_normal((8, 512)) * 1e-30).astype(np.float32)


@pytest.mark.parametrize("name,x", list(_dists()))
def test_quantize_invariants(oracle, name, x):
    q, s = oracle.quantize_rows(x)
    assert q.dtype == np.int8 and s.dtype == np.float32
    assert np.all(np.abs(q.astype(np.int32)) <= 127)          # -128 never produced
    assert np.all(np.isfinite(s)) and np.all(s > 0)           # finite positive scales
    # the absmax element of each row maps to +-127 with its sign
    idx = np.argmax(np.abs(x), axis=1)
    ar = np.arange(x.shape[0])
    assert np.all(q[ar, idx] == np.sign(x[ar, idx]).astype(np.int8) * 127)
    # reconstruction error at most half a step (plus FP32 slack)
    err = np.abs(x.astype(np.float64) - s[:, None].astype(np.float64) * q)
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-5))
    # odd symmetry
    qn, sn = oracle.quantize_rows(-x)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    # power-of-two scaling leaves q unchanged and scales s exactly
    if name != "tiny":
        q2, s2 = oracle.quantize_rows(x * np.float32(8.0))
        assert np.array_equal(q2, q) and np.array_equal(s2, s * np.float32(8.0))


def test_quantize_zero_and_constant_rows(oracle):
    x = np.zeros((3, 64), np.float32)
    x[1, :] = 0.75
    x[2, :] = -3.0e-5
    q, s = oracle.quantize_rows(x)
    assert s[0] == 1.0 and np.all(q[0] == 0)
    assert np.all(q[1] == 127) and np.all(q[2] == -127)


def test_quantize_rejects_non_finite(oracle):
    for bad in (np.inf, -np.inf, np.nan):
        x = np.ones((2, 16), np.float32)
        x[1, 5] = bad
        with pytest.raises(ValueError):
            oracle.quantize_rows(x)


def test_quantize_act_widens_bf16_exactly(oracle):
    # BF16 bit patterns of +-1.5, 0, 3.0, 2^-133 (smallest subnormal)
    bits = np.array([[0x3FC0, 0xBFC0, 0x0000, 0x4040, 0x0001]], np.uint16)
    x = oracle.widen_bf16(bits)
    assert x.tolist() == [[1.5, -1.5, 0.0, 3.0, 2.0 ** -133]]
    q, s = oracle.quantize_act(bits)
    assert q[0].tolist() == [64, -64, 0, 127, 0]   # 1.5/(3/127) is 63.5 within FP32 rounding -> 64
    assert float(s[0]) == float(np.float32(3.0) / np.float32(127.0))


def test_bf16_subnormal_row_keeps_positive_scale(oracle):
    bits = np.array([[0x0001, 0x8001, 0x0000]], np.uint16)   # +-2^-133
    q, s = oracle.quantize_act(bits)
    assert s[0] > 0 and q[0].tolist() == [127, -127, 0]


# --- INT32 GEMM --------------------------------------------------------------------

def test_gemm_python_int_brute_force(oracle):
    rng = np.random.default_rng(3)
    for M, N, K in [(1, 1, 16), (3, 5, 48), (7, 4, 64), (5, 9, 130)]:
        qa = rng.integers(-127, 128, (M, K), dtype=np.int8)
        qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
        acc = oracle.gemm_int32(qa, qw)
        for m in range(M):
            for n in range(N):
                assert int(acc[m, n]) == sum(int(qa[m, k]) * int(qw[n, k]) for k in range(K))


@pytest.mark.parametrize("K,expect", [(5376, 86_709_504), (21504, 346_838_016)])
def test_gemm_closed_form_all_127(oracle, K, expect):
    qa = np.full((2, K), 127, np.int8)
    qw = np.full((3, K), 127, np.int8)
    qw[1] = -127
    acc = oracle.gemm_int32(qa, qw)
    assert acc[:, 0].tolist() == [expect, expect]
    assert acc[:, 1].tolist() == [-expect, -expect]


def test_gemm_unit_vectors_pick_weight_columns(oracle):
    rng = np.random.default_rng(9)
    K, N = 96, 7
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    qa = np.zeros((K, K), np.int8)
    np.fill_diagonal(qa, 1)
    qa[5, 5] = -1
    acc = oracle.gemm_int32(qa, qw)
    expect = qw.T.astype(np.int32).copy()
    expect[5] *= -1
    assert np.array_equal(acc, expect)          # catches a transposed operand


def test_gemm_partial_sums_cross_2_pow_24(oracle):
    # alternating blocks whose running sums exceed 2^24 before cancelling: an
    # FP32 accumulator would lose bits here, INT32 must not
    K = 5376
    qa = np.full((1, K), 127, np.int8)
    qw = np.full((2, K), 127, np.int8)
    qw[0, K // 2:] = -127
    qw[0, -1] = 126
    qw[1, ::2] = 1
    acc = oracle.gemm_int32(qa, qw)
    # 2688 terms of +127^2, 2687 of -127^2, one of 127*126
    assert int(acc[0, 0]) == (K // 2) * 127 * 127 - (K // 2 - 1) * 127 * 127 + 127 * 126
    assert int(acc[0, 1]) == (K // 2) * 127 + (K // 2) * 127 * 127


# --- BF16 rounding and the epilogue -------------------------------------------------

def test_round_to_bf16_hand_cases(oracle):
    for c in _load("bf16_round_cases.json")["cases"]:
        num, p = c["v"]
        v = math.ldexp(float(num), p)
        assert int(oracle.round_to_bf16(np.array([v]))[0]) == int(c["bits"], 16), c["why"]


def test_round_to_bf16_matches_torch_on_fp32_values(oracle):
    # special case that reduces to a library routine: for a float64 that is an
    # exact FP32 value, one rounding to BF16 is torch's FP32 -> BF16 cast
    import torch
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),      # subnormals
        (rng.standard_normal(2000) * 1e38).astype(np.float32),
        # exact BF16 ties: a BF16 value plus half its spacing
        (np.arange(1, 2001, dtype=np.float32) * np.float32(2.0 ** -7) + np.float32(1.0)
         + np.float32(2.0 ** -8)),
    ])
    got = oracle.round_to_bf16(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_epilogue_golden_cases(oracle):
    for c in _load("epilogue_cases.json")["cases"]:
        acc = np.array([[c["acc"]]], np.int32)
        sa = np.array([c["s_a"]], np.float32)
        sw = np.array([c["s_w"]], np.float32)
        bias = None if c["bias_bits"] is None else np.array([int(c["bias_bits"], 16)], np.uint16)
        y = oracle.round_to_bf16(oracle.epilogue_value(acc, sa, sw, bias))
        assert int(y[0, 0]) == int(c["y_bits"], 16), c["name"]


def test_linear_zero_rows_give_bias_or_zero(oracle):
    rng = np.random.default_rng(2)
    K, N = 64, 16
    x = np.zeros((3, K), np.uint16)
    x[1] = 0x8000                        # -0.0 everywhere: still an all-zero row
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qw, sw = oracle.quantize_weights(w)
    bias = np.array([0x3F80 + i for i in range(N)], np.uint16)
    out = oracle.linear(x, qw, sw, bias)
    assert np.all(out["acc"] == 0) and np.all(out["sa"] == 1.0)
    assert np.all(out["y"] == bias[None, :])
    out0 = oracle.linear(x, qw, sw, None)
    assert np.all((out0["y"] & 0x7FFF) == 0)


def test_linear_matches_unquantised_product_roughly(oracle):
    # sanity, not parity: W8A8 tracks the FP32 matmul (signal-to-noise > 30 dB)
    rng = np.random.default_rng(4)
    import synth
    x = rng.standard_normal((32, 512)).astype(np.float32)
    xb = synth.to_bf16_bits(x)
    w = (rng.standard_normal((48, 512)) * 0.02).astype(np.float32)
    qw, sw = oracle.quantize_weights(w)
    out = oracle.linear(xb, qw, sw, None)
    ref = oracle.widen_bf16(xb).astype(np.float64) @ w.astype(np.float64).T
    snr = 10 * np.log10(np.sum(ref ** 2) / np.sum((out["v"] - ref) ** 2))
    assert snr > 30


# --- converter scope rule: passthrough -------------------------------------------

def test_converter_passthrough_is_byte_identical(oracle):
    rng = np.random.default_rng(8)
    tensors = {}
    for b in range(3):
        for p in ("attn.to_q", "attn.to_k", "attn.to_v", "attn.to_out", "mlp.fc1", "mlp.fc2",
                  "adaln.linear", "norm1"):
            tensors[f"blocks.{b}.{p}.weight"] = rng.standard_normal((8, 32)).astype(np.float32)
        tensors[f"blocks.{b}.attn.to_q.bias"] = rng.standard_normal(8).astype(np.float32)
    tensors["text_encoder.embed.weight"] = rng.standard_normal((16, 32)).astype(np.float32)
    tensors["vae.decoder.conv.weight"] = np.arange(20, dtype=np.uint16)
    h = {k: hashlib.sha256(v.tobytes()).hexdigest() for k, v in tensors.items()}

    for profile, n_quant in (("dit_proj", 18), ("mlp", 6)):
        out = oracle.convert_state_dict(tensors, profile=profile, n_blocks=3)
        quantised = [k for k in tensors if oracle.in_scope(k, profile, 3)]
        assert len(quantised) == n_quant
        for k, v in tensors.items():
            if k in quantised:
                assert out[k].dtype == np.int8
                s = out[k[:-len(".weight")] + ".weight_scale"]
                assert s.dtype == np.float32 and np.all(np.isfinite(s)) and np.all(s > 0)
            else:
                assert hashlib.sha256(out[k].tobytes()).hexdigest() == h[k]
                assert out[k].dtype == v.dtype and out[k].shape == v.shape
        assert len(out) == len(tensors) + n_quant


# --- accuracy report: the unquantised reference Linear and the SNR ----------------

def test_reference_linear_brute_force(oracle):
    rng = np.random.default_rng(90)
    M, N, K = 3, 4, 5
    xb = oracle.round_to_bf16(rng.standard_normal((M, K)))
    w = rng.standard_normal((N, K)).astype(np.float32)
    bb = oracle.round_to_bf16(rng.standard_normal(N))
    x = oracle.widen_bf16(xb)
    b = oracle.widen_bf16(bb)
    ref = oracle.reference_linear(xb, w, bb)
    for m in range(M):
        for n in range(N):
            # exact rational sum of products of the FP32 values, then the bias
            exact = sum(Fraction(float(x[m, k])) * Fraction(float(w[n, k])) for k in range(K))
            exact += Fraction(float(b[n]))
            assert abs(ref[m, n] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))
    assert np.array_equal(oracle.reference_linear(xb, w), ref - b)


def test_snr_closed_forms(oracle):
    rng = np.random.default_rng(91)
    ref = rng.standard_normal(1000)
    assert oracle.snr_db(ref, ref) == float("inf")
    assert abs(oracle.snr_db(np.zeros_like(ref), ref) - 0.0) < 1e-12
    # a uniform 1 % relative error is 40 dB; a 10 % one is 20 dB
    assert abs(oracle.snr_db(ref * 1.01, ref) - 40.0) < 1e-9
    assert abs(oracle.snr_db(ref * 0.9, ref) - 20.0) < 1e-9
    # halving the noise amplitude gains 20 log10(2) dB
    noise = rng.standard_normal(1000) * 1e-3
    d = oracle.snr_db(ref + noise / 2, ref) - oracle.snr_db(ref + noise, ref)
    assert abs(d - 20 * np.log10(2)) < 1e-9


# --- the group-wise affine comparison scheme (readings R10-R13) ------------------
# "MLX implementation and experiment report", Operator tuning (Q8/g64, Q4/g64);
# "[feat] Add MiniMax H3 MLX T2VA inference" (affine INT8/INT6/INT4 checkpoints).

def _brute_affine_group(ws, bits):
    ws = [Fraction(float(v)) for v in ws]
    lo, hi = min(ws), max(ws)
    levels = 2 ** bits - 1
    if hi == lo:
        alpha = Fraction(1)
    else:
        alpha = _fp32_rn(_fp32_rn(hi - lo) / levels)
    q = [max(0, min(levels, _rne_int(_fp32_rn(_fp32_rn(v - lo) / alpha)))) for v in ws]
    return q, alpha, lo


@pytest.mark.parametrize("bits", [8, 4])
def test_affine_brute_force_rationals(oracle, bits):
    rng = np.random.default_rng(40 + bits)
    w = (rng.standard_normal((3, 128)) * 0.05).astype(np.float32)
    w[1, 64:] = np.float32(0.25)                       # a constant group
    q, a, b = oracle.quantize_affine(w, bits=bits)
    for n in range(3):
        for g in range(2):
            bq, ba, bb = _brute_affine_group(w[n, 64 * g:64 * g + 64], bits)
            assert list(q[n, 64 * g:64 * g + 64]) == bq
            assert Fraction(float(a[n, g])) == ba and Fraction(float(b[n, g])) == bb


def test_affine_grid_reconstructs_exactly(oracle):
    # values beta + j / 64 for j in 0..255 (both ends present): alpha comes out
    # as exactly 1/64, q = j, and the dequantised weights are the inputs
    rng = np.random.default_rng(44)
    j = rng.integers(0, 256, (4, 256))
    j[:, ::64] = 0
    j[:, 1::64] = 255
    w = (np.float32(-0.5) + j.astype(np.float32) / np.float32(64.0)).astype(np.float32)
    q, a, b = oracle.quantize_affine(w, bits=8)
    assert np.array_equal(q, j.astype(np.uint8))
    assert np.all(a == np.float32(1 / 64)) and np.all(b == np.float32(-0.5))
    wh = oracle.dequant_affine(q, a, b)
    assert np.array_equal(oracle.widen_bf16(wh), w)       # every such value is a BF16 value


def test_affine_4bit_grid_reconstructs_exactly(oracle):
    # the 4-bit case of the grid above: beta + j / 16 for j in 0..15 (both
    # ends present) gives alpha = (15/16) / 15 = 1/16 exactly, q = j, and
    # dequantised weights equal to the inputs
    rng = np.random.default_rng(46)
    j = rng.integers(0, 16, (4, 128))
    j[:, ::64] = 0
    j[:, 1::64] = 15
    w = (np.float32(0.25) + j.astype(np.float32) / np.float32(16.0)).astype(np.float32)
    q, a, b = oracle.quantize_affine(w, bits=4)
    assert np.array_equal(q, j.astype(np.uint8))
    assert np.all(a == np.float32(1 / 16)) and np.all(b == np.float32(0.25))
    assert np.array_equal(oracle.widen_bf16(oracle.dequant_affine(q, a, b)), w)


@pytest.mark.parametrize("bits", [8, 4])
def test_affine_extremes_and_error_bound(oracle, bits):
    rng = np.random.default_rng(45 + bits)
    w = (rng.standard_normal((16, 512)) * 0.02).astype(np.float32)
    q, a, b = oracle.quantize_affine(w, bits=bits)
    g = w.reshape(16, 8, 64)
    qg = q.reshape(16, 8, 64)
    # the group's minimum codes to 0 and its maximum to 2^bits - 1
    assert np.all(np.take_along_axis(qg, g.argmin(2)[:, :, None], 2) == 0)
    assert np.all(np.take_along_axis(qg, g.argmax(2)[:, :, None], 2) == 2 ** bits - 1)
    # rint: |w - (alpha q + beta)| <= alpha / 2, up to the FP32 roundings
    rec = qg.astype(np.float64) * a[:, :, None] + b[:, :, None]
    assert np.all(np.abs(g - rec) <= a[:, :, None] * (0.5 + 2.0 ** -10))


def test_affine_constant_group_and_rejects_non_finite(oracle):
    w = np.full((2, 64), -0.375, np.float32)
    q, a, b = oracle.quantize_affine(w)
    assert np.all(q == 0) and np.all(a == 1.0) and np.all(b == np.float32(-0.375))
    assert np.all(oracle.widen_bf16(oracle.dequant_affine(q, a, b)) == np.float32(-0.375))
    w[1, 7] = np.nan
    with pytest.raises(ValueError):
        oracle.quantize_affine(w)


def test_dequant_affine_one_fp32_rounding_then_bf16(oracle):
    # brute force: RN_fp32(alpha q + beta) in rationals, then one BF16 rounding;
    # the last group has beta far above alpha q, where the float64 sum itself
    # rounds and the oracle takes its exact-rational path
    rng = np.random.default_rng(47)
    q = rng.integers(0, 256, (2, 128)).astype(np.uint8)
    a = (rng.uniform(1e-4, 1e-2, (2, 2))).astype(np.float32)
    b = (rng.uniform(-0.5, 0.5, (2, 2))).astype(np.float32)
    a[1, 1] = np.float32(2.0 ** -40)
    b[1, 1] = np.float32(2.0 ** 30 + 2.0 ** 7)
    wh = oracle.dequant_affine(q, a, b)
    for n in range(2):
        for k in range(128):
            g = k // 64
            v = _fp32_rn(Fraction(int(q[n, k])) * Fraction(float(a[n, g])) +
                         Fraction(float(b[n, g])))
            want = oracle.round_to_bf16(np.array([float(v)], np.float64))[0]
            assert wh[n, k] == want, (n, k)


def test_linear_affine_brute_force(oracle):
    rng = np.random.default_rng(48)
    xb = oracle.round_to_bf16(rng.standard_normal((3, 128)))
    wb = oracle.round_to_bf16(rng.standard_normal((5, 128)) * 0.1)
    bias = oracle.round_to_bf16(rng.standard_normal(5))
    out = oracle.linear_affine(xb, wb, bias)
    xf, wf = oracle.widen_bf16(xb), oracle.widen_bf16(wb)
    bf = oracle.widen_bf16(bias)
    for m in range(3):
        for n in range(5):
            exact = sum(Fraction(float(xf[m, k])) * Fraction(float(wf[n, k])) for k in range(128))
            exact += Fraction(float(bf[n]))
            assert abs(Fraction(float(out["v"][m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 50)
            assert out["absum"][m, n] == pytest.approx(
                float(sum(abs(Fraction(float(xf[m, k])) * Fraction(float(wf[n, k])))
                          for k in range(128))), rel=1e-12)


def test_affine_q8_beats_q4(oracle):
    # more levels, smaller steps: the 8-bit reconstruction error is below the
    # 4-bit one by about the ratio of the steps (255 / 15 = 17)
    rng = np.random.default_rng(49)
    w = (rng.standard_normal((64, 1024)) * 0.02).astype(np.float32)
    err = {}
    for bits in (8, 4):
        q, a, b = oracle.quantize_affine(w, bits=bits)
        rec = (q.reshape(64, 16, 64).astype(np.float64) * a[:, :, None] + b[:, :, None])
        err[bits] = float(np.sqrt(np.mean((rec.reshape(64, 1024) - w) ** 2)))
    assert 12 < err[4] / err[8] < 22
