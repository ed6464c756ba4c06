"""CPU oracle for the W8A8 INT8 projection Linear.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never calls it, shares
no code with it, and fails loudly when it is missing; this file exists to say
what the right answer is, slowly and plainly, in numpy.

Sources (cited by page title and section):
  [P1] "feat(mps): support MiniMax-H3 INT8 inference on Apple M5"
       (ModelTC/LightX2V pull request #1672).
  [P2] "MLX implementation and experiment report"
       (MiniMax-H3-Image-mlx, reports/RESULTS.md).
  [P4] "[feat] Add MiniMax H3 MLX T2VA inference"
       (hao-ai-lab/FastVideo pull request #1770).

What the pages fix: pre-quantised W8A8 projections at the native width K=5376
with no K padding and no weight dequantisation ([P1] opening description);
INT8 weights with finite positive FP32 per-channel scales, produced by a
per-row converter that leaves every other tensor byte-for-byte unchanged
([P1] Validation; Changes table, row "Quantization scopes and checkpoint
conversion"); a per-token activation quantiser with masked tail chunks
([P1] Summary by CodeRabbit; Changes table, row "INT8 Metal GEMM shapes and
execution"); CPU INT32 references for the INT8 product ([P1] Validation);
and a biased BF16 Linear whose bias is added before the one rounding of the
output ([P2] What the default preserves, the "addmm epilogue" bullet).

The pages print no formula for the quantiser or the epilogue.  The readings
taken where they are silent:
  R1  scale = absmax / 127 as one IEEE FP32 division, round to nearest even;
  R2  q = clamp(rint(x / scale), -127, 127): FP32 division by the scale (not a
      multiply by 127/absmax), ties to even, -128 never produced;
  R3  an all-zero row gets scale 1.0 and q = 0 (the only finite positive
      scale that leaves the row exactly representable); a non-zero row whose
      absmax/127 underflows to +0 gets the smallest positive FP32 (2^-149);
  R4  non-finite inputs are rejected (scales must be finite and positive);
  R5  the epilogue value is v = acc * s_a[m] * s_w[n] + bias[n], evaluated here
      in float64 from the exact INT32 accumulator and the FP32 scales, and the
      BF16 output is v rounded once to nearest even; a GPU result is accepted
      within one BF16 ulp of v (the order of the FP32 operations on the GPU is
      not fixed by the pages);
  R6  masked tail chunks change nothing in the result: the quantiser is
      defined per row over exactly K elements.

The group-wise affine scheme of [P2] and [P4] (weights only), a comparison
point for the W8A8 path, has readings R10-R13 below, with its functions.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import re

import numpy as np

QMAX = 127
_SMALLEST_F32 = np.float32(np.finfo(np.float32).smallest_subnormal)


# --- BF16 <-> FP32/FP64 --------------------------------------------------------

def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32, exactly (BF16 is the top half of FP32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """float64 -> BF16 bit patterns, one rounding to nearest, ties to even.

    Written from the IEEE-754 definition of the binary16-brain format: 8
    significant bits, FP32's exponent range (normal exponents -126..127),
    subnormal spacing 2^-133, overflow to infinity at or above the halfway
    point past the largest finite value.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    sign = np.signbit(v).astype(np.uint16) << 15
    a = np.abs(v)
    nan = np.isnan(a)
    with np.errstate(invalid="ignore", over="ignore"):
        fin = np.isfinite(a)
        m, e = np.frexp(np.where(fin, a, 0.0))          # a = m * 2^e, m in [0.5, 1)
        unbiased = e - 1                                 # a = 1.f * 2^unbiased
        q_exp = np.where(unbiased < -126, -133, unbiased - 7)   # spacing of BF16 here
        n = np.rint(np.ldexp(np.where(fin, a, 0.0), -q_exp))     # exact scaling, RNE
        r = np.ldexp(n, q_exp)                           # a BF16 value, or >= 2^128
        over = (r >= 2.0 ** 128) | ~fin
        r32 = np.where(over, 0.0, r).astype(np.float32)  # exact: r is a BF16 value
        mag = (r32.view(np.uint32) >> 16).astype(np.uint16)
    mag = np.where(over, np.uint16(0x7F80), mag)
    out[...] = sign | mag
    out[nan] = 0x7FC0
    return out


# --- A1 / A2: symmetric per-row INT8 quantisation --------------------------------

def quantize_rows(x: np.ndarray):
    """Quantise each row of ``x`` (float32 [R, K]) to INT8 with one FP32 scale.

    For a weight matrix the rows are output channels ([P1] Validation:
    "INT8 weights and finite positive FP32 per-channel scales"; Changes table,
    "per-row INT8 conversion"); for activations they are tokens ([P1] Changes
    table, "INT8 Metal GEMM shapes and execution": the activation quantiser).
    Readings R1-R4 and R6 of the module docstring apply.

    Returns (q int8 [R, K], scale float32 [R]).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("quantize_rows expects a 2-D array")
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite input: scales must be finite and positive (R4)")
    a = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = a / np.float32(QMAX)                                     # R1: one FP32 division
    s = np.where(a == 0, np.float32(1.0), s)                     # R3: zero row
    s = np.where((a > 0) & (s == 0), _SMALLEST_F32, s).astype(np.float32)  # R3: underflow
    r = x / s[:, None]                                           # R2: FP32 division
    q = np.clip(np.rint(r), -QMAX, QMAX).astype(np.int8)         # R2: RNE, clamp
    return q, s


def quantize_weights(w: np.ndarray):
    """A1: FP32 (or BF16 bits, widened exactly) weight [N, K] -> (int8, FP32 scale)."""
    w = np.asarray(w)
    if w.dtype == np.uint16:
        w = widen_bf16(w)
    return quantize_rows(w)


def quantize_act(x_bits: np.ndarray):
    """A2: BF16 activations [M, K] (bit patterns) -> (int8, FP32 scale) per token."""
    return quantize_rows(widen_bf16(x_bits))


# --- A3: INT8 x INT8 -> INT32 -------------------------------------------------

def gemm_int32(qa: np.ndarray, qw: np.ndarray) -> np.ndarray:
    """acc[m, n] = sum_k qa[m, k] * qw[n, k], in INT32 ([P1] Validation: "CPU INT32
    references for native INT8 output").

    The product is taken as a float64 matrix product of the integer values:
    every partial sum is an integer no larger than K * 127^2 < 2^53, so each
    one is exact in float64 whatever order the library sums in.
    """
    qa = np.asarray(qa, dtype=np.int8)
    qw = np.asarray(qw, dtype=np.int8)
    if qa.shape[1] != qw.shape[1]:
        raise ValueError("K mismatch")
    K = qa.shape[1]
    if K * QMAX * QMAX >= 2 ** 53:
        raise ValueError("K too large for an exact float64 product")
    acc = qa.astype(np.float64) @ qw.astype(np.float64).T
    if acc.size and np.max(np.abs(acc)) >= 2 ** 31:
        raise OverflowError("INT32 accumulator overflow")
    return acc.astype(np.int32)


# --- A4: dequantise + bias + one BF16 rounding -----------------------------------

def epilogue_value(acc, sa, sw, bias_bits=None) -> np.ndarray:
    """v[m, n] = acc[m, n] * s_a[m] * s_w[n] + bias[n], in float64 (reading R5).

    The bias is added before the single rounding to BF16 ([P2] What the default
    preserves: biased BF16 linears use an addmm epilogue; rounding the product
    first and then adding the bias changes results).
    """
    v = (np.asarray(acc, dtype=np.float64)
         * np.asarray(sa, dtype=np.float64)[:, None]
         * np.asarray(sw, dtype=np.float64)[None, :])
    if bias_bits is not None:
        v = v + widen_bf16(bias_bits).astype(np.float64)[None, :]
    return v


def linear(x_bits, qw, sw, bias_bits=None) -> dict:
    """The whole hot path for one Linear: A2, A3, A4.

    Returns a dict with the INT8 activations ``qa``, their scales ``sa``, the
    INT32 accumulator ``acc``, the float64 epilogue value ``v`` and the BF16
    output bits ``y``.
    """
    qa, sa = quantize_act(x_bits)
    acc = gemm_int32(qa, qw)
    v = epilogue_value(acc, sa, sw, bias_bits)
    return {"qa": qa, "sa": sa, "acc": acc, "v": v, "y": round_to_bf16(v)}


# --- accuracy of the quantised Linear against the unquantised one --------------------
# [P4] review notes, test coverage: an INT8 SNR check.  The pages give no
# formula; the plain reading: the unquantised Linear y_ref = X W^T + bias
# (BF16 X and bias widened exactly, FP32 W) evaluated in float64, and
#   SNR = 10 log10( sum y_ref^2 / sum (y - y_ref)^2 )  dB
# for the quantised outputs y over the same elements.

def reference_linear(x_bits, w, bias_bits=None) -> np.ndarray:
    """The unquantised Linear in float64: widen(X) @ W^T + widen(bias)."""
    y = widen_bf16(x_bits).astype(np.float64) @ np.asarray(w, dtype=np.float64).T
    if bias_bits is not None:
        y = y + widen_bf16(bias_bits).astype(np.float64)
    return y


def snr_db(y, y_ref) -> float:
    """Signal-to-noise ratio of y against y_ref, in dB (inf when equal)."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    noise = float(np.sum((y - y_ref) ** 2))
    signal = float(np.sum(y_ref ** 2))
    if noise == 0.0:
        return float("inf")
    return 10.0 * np.log10(signal / noise)


# --- the comparison scheme: group-wise affine weight-only quantisation ---------------
# [P2] Operator tuning times Q8/g64 and Q4/g64 variants of the QKV, gate/up and
# down GEMMs; [P4] adds affine INT8, INT6 and INT4 checkpoints.  That scheme is
# weight-only: per output channel and group of 64 consecutive inputs a step and
# an offset ("affine"), the weights dequantised for a BF16 GEMM with the BF16
# activations unquantised.  The pages give no formula; the readings:
#   R10  per group: lo = min, hi = max of its FP32 weights; alpha = RN((hi - lo)
#       / (2^b - 1)), hi - lo rounded to FP32 first, one FP32 division;
#       beta = lo; a group with hi == lo gets alpha = 1, and a positive range
#       whose alpha underflows to 0 gets the smallest positive FP32;
#   R11  q = clamp(rint(RN(RN(w - beta) / alpha)), 0, 2^b - 1): FP32 subtraction
#       and division, ties to even;
#   R12  the dequantised weight is w^ = BF16_RNE(RN_fp32(alpha q + beta)): one
#       FP32 fused multiply-add, then BF16, the activations' type (a tensor-core
#       MMA takes both operands in one type);
#   R13 y = BF16_RNE(sum_k x_k w^_k + bias): the reference sum is evaluated in
#       float64 (the products are exact), and a GPU result, whose FP32
#       accumulation order is not fixed, is accepted within one BF16 ulp plus
#       K 2^-23 sum_k |x_k w^_k|.

AFFINE_GROUP = 64


def quantize_affine(w: np.ndarray, bits: int = 8, group: int = AFFINE_GROUP):
    """Group-wise affine quantisation of a weight [N, K] (FP32, or BF16 bits
    widened exactly), K a multiple of ``group``; readings R10, R11.

    Returns (q uint8 [N, K] in [0, 2^bits - 1], alpha float32 [N, K/group],
    beta float32 [N, K/group]).
    """
    w = np.asarray(w)
    if w.dtype == np.uint16:
        w = widen_bf16(w)
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    if k % group:
        raise ValueError("K must be a multiple of the group size")
    if not np.all(np.isfinite(w)):
        raise ValueError("non-finite weight")
    g = w.reshape(n, k // group, group)
    lo = g.min(axis=2)
    hi = g.max(axis=2)
    levels = np.float32(2 ** bits - 1)
    alpha = (hi - lo) / levels                                    # FP32 ops, RN
    alpha = np.where(hi == lo, np.float32(1.0), alpha)
    alpha = np.where((hi > lo) & (alpha == 0), _SMALLEST_F32, alpha).astype(np.float32)
    beta = lo.astype(np.float32)
    d = g - beta[:, :, None]                                      # FP32 subtraction
    r = d / alpha[:, :, None]                                     # FP32 division
    q = np.clip(np.rint(r), 0, levels).astype(np.uint8)
    return q.reshape(n, k), alpha, beta


def _exact_sum_or_none(a: np.ndarray, b: np.ndarray):
    """a + b in float64 and a mask of the elements where that sum rounded
    (Knuth's two-sum error term is non-zero)."""
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)
    return s, err != 0


def dequant_affine(q: np.ndarray, alpha: np.ndarray, beta: np.ndarray,
                   group: int = AFFINE_GROUP) -> np.ndarray:
    """R12: w^ = BF16_RNE(RN_fp32(alpha q + beta)) as BF16 bit patterns [N, K]."""
    n, k = q.shape
    qq = q.reshape(n, k // group, group).astype(np.float64)
    a = alpha.astype(np.float64)[:, :, None]
    b = beta.astype(np.float64)[:, :, None]
    prod = qq * a                                   # exact: 24 + 8 significant bits
    exact, rounded = _exact_sum_or_none(prod, np.broadcast_to(b, prod.shape))
    if np.any(rounded):
        # the float64 sum rounded (operands far apart in magnitude): redo those
        # elements in exact rational arithmetic, then round to FP32 once
        from fractions import Fraction
        idx = np.argwhere(rounded)
        for (i, j, t) in idx:
            v = Fraction(float(qq[i, j, t])) * Fraction(float(a[i, j, 0])) + \
                Fraction(float(b[i, j, 0]))
            exact[i, j, t] = _fraction_to_f32(v)
    f32 = exact.astype(np.float32)                  # RN to FP32 (exact cases: one rounding)
    return round_to_bf16(f32.reshape(n, k))


def _fraction_to_f32(v) -> float:
    """Round an exact rational to the nearest FP32 (ties to even), as a float."""
    import math
    if v == 0:
        return 0.0
    sign = -1.0 if v < 0 else 1.0
    v = abs(v)
    e = math.floor(math.log2(v.numerator) - math.log2(v.denominator))
    while 2 ** e > v:
        e -= 1
    while 2 ** (e + 1) <= v:
        e += 1
    q_exp = max(e, -126) - 23                      # FP32 spacing at this magnitude
    from fractions import Fraction
    scaled = v / Fraction(2) ** q_exp
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * float(Fraction(n) * Fraction(2) ** q_exp)


def linear_affine(x_bits: np.ndarray, w_hat_bits: np.ndarray, bias_bits=None) -> dict:
    """R13: the weight-only Linear on dequantised BF16 weights.  Returns the
    float64 value v, sum_k |x_k w^_k| (for the tolerance) and y = BF16_RNE(v)."""
    xf = widen_bf16(x_bits).astype(np.float64)
    wf = widen_bf16(w_hat_bits).astype(np.float64)
    v = xf @ wf.T
    if bias_bits is not None:
        v = v + widen_bf16(bias_bits).astype(np.float64)
    return {"v": v, "absum": np.abs(xf) @ np.abs(wf).T, "y": round_to_bf16(v)}


# --- the converter's scope rule (passthrough) -------------------------------------

# Per-block projection names of the dit_proj profile: Q, K, V, attention output,
# FC1 and FC2 ([P1] opening description).  The pages give no tensor names; these
# are synthetic stand-ins.
PROFILES = {
    "dit_proj": ("attn.to_q", "attn.to_k", "attn.to_v", "attn.to_out", "mlp.fc1", "mlp.fc2"),
    "mlp": ("mlp.fc1", "mlp.fc2"),
}
_BLOCK_RE = re.compile(r"^blocks\.(\d+)\.(.+)\.weight$")


def in_scope(name: str, profile: str = "dit_proj", n_blocks: int = 50) -> bool:
    m = _BLOCK_RE.match(name)
    return bool(m) and int(m.group(1)) < n_blocks and m.group(2) in PROFILES[profile]


def convert_state_dict(tensors: dict, profile: str = "dit_proj", n_blocks: int = 50) -> dict:
    """Quantise the in-scope projection weights; pass every other tensor through.

    [P1] Validation: the standalone conversion kept all unquantised tensors
    byte-for-byte and produced INT8 weights with finite positive FP32
    per-channel scales.  In-scope ``<name>.weight`` becomes INT8 and gains
    ``<name>.weight_scale``; everything else is returned unchanged (the same
    bytes).
    """
    out = {}
    for name, t in tensors.items():
        if in_scope(name, profile, n_blocks):
            q, s = quantize_weights(t)
            out[name] = q
            out[name[: -len(".weight")] + ".weight_scale"] = s
        else:
            out[name] = t
    return out
