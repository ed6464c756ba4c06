"""Comparison helpers for GPU-vs-oracle parity (test-side only).

The bar: INT8 activations, FP32 scales and INT32 accumulators bit-exact; the
BF16 output within one BF16 ulp of the oracle's float64 epilogue value v,
where ulp(v) is the spacing of BF16 numbers in the binade of |v|
(2^(floor(log2|v|) - 7), and 2^-133 below the normal range).
"""
import numpy as np


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)
    unbiased = np.where(a > 0, e - 1, -126)
    return np.ldexp(1.0, np.maximum(unbiased, -126) - 7)


def widen(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# |v| at or above this rounds to infinity in BF16: (2 - 2^-8) * 2^127
BF16_OVERFLOW = (2.0 - 2.0 ** -8) * 2.0 ** 127


def check_y(y_bits: np.ndarray, v: np.ndarray, what: str = "y") -> dict:
    """Assert |y - v| <= 1 BF16 ulp(v) everywhere (and y = +-inf exactly where v
    itself overflows BF16); return match statistics."""
    y = widen(y_bits).astype(np.float64)
    v = np.asarray(v, dtype=np.float64)
    over = np.abs(v) >= BF16_OVERFLOW
    if np.any(over):
        assert np.array_equal(y[over], np.copysign(np.inf, v[over])), f"{what}: overflow mismatch"
        y = np.where(over, 0.0, y)
        v = np.where(over, 0.0, v)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output where the exact value is finite"
    err = np.abs(y - v)
    ulp = bf16_ulp(v)
    ratio = err / ulp
    worst = float(ratio.max()) if ratio.size else 0.0
    bad = np.argwhere(ratio > 1.0)
    assert bad.size == 0, (f"{what}: {len(bad)} outputs beyond 1 BF16 ulp, first at "
                           f"{tuple(bad[0])}: y={y[tuple(bad[0])]!r} v={v[tuple(bad[0])]!r}")
    return {"max_ulp": worst}


def check_exact(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    if got.dtype.kind == "f":
        eq = got.view(np.uint32 if got.itemsize == 4 else np.uint64) == \
            want.astype(got.dtype).view(np.uint32 if got.itemsize == 4 else np.uint64)
    else:
        eq = got == want
    if not np.all(eq):
        idx = tuple(np.argwhere(~eq)[0])
        raise AssertionError(f"{what}: {int((~eq).sum())} mismatches, first at {idx}: "
                             f"got {got[idx]!r} want {want[idx]!r}")
