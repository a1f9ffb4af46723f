"""Comparison rules between the CUDA path and the oracle.

* bf16 outputs: the CUDA result must be within 1 bf16 ulp of the oracle's fp64 result
  rounded once (round to nearest even). Distance is measured in ordinal steps of the
  bf16 encoding; +0 and -0 are the same point.
* fp16 outputs: the same rule in binary16 (1 ulp of the oracle's fp64 result rounded
  once). The kernels compute in fp32 (relative error a few times 2^-24 on these
  operators, RoPE's compensated products included) and round once, so the result is
  the correctly rounded value or, when the fp32 value lies within that error of a
  rounding boundary, its neighbour.
* fp32 outputs: |got - ref| <= 1e-6 + 2e-6 * |ref| against the oracle's unrounded fp64
  result.
"""

from __future__ import annotations

import numpy as np

FP32_ATOL = 1e-6
FP32_RTOL = 2e-6
BF16_MAX_ULPS = 1
F16_MAX_ULPS = 1

DTYPES = ["bf16", "f16", "f32"]
ES = {"bf16": 2, "f16": 2, "f32": 4}   # bytes per element


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that are monotonic in value (+0 == -0 == 0)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(bf16_ordinal(a_bits) - bf16_ordinal(b_bits))


def assert_bf16_close(got_bits: np.ndarray, want_bits: np.ndarray, what: str = "") -> None:
    got_bits = np.asarray(got_bits)
    want_bits = np.asarray(want_bits)
    assert got_bits.shape == want_bits.shape, (got_bits.shape, want_bits.shape)
    if got_bits.size == 0:
        return
    d = bf16_ulp_distance(got_bits, want_bits)
    worst = int(d.max())
    if worst > BF16_MAX_ULPS:
        idx = np.unravel_index(int(d.argmax()), d.shape)
        n_bad = int((d > BF16_MAX_ULPS).sum())
        raise AssertionError(
            f"{what}: {n_bad} bf16 outputs beyond {BF16_MAX_ULPS} ulp; worst {worst} ulp at "
            f"{idx}: got 0x{int(got_bits[idx]):04x}, want 0x{int(want_bits[idx]):04x}")


def assert_f32_close(got: np.ndarray, ref64: np.ndarray, what: str = "") -> None:
    got = np.asarray(got, dtype=np.float32).astype(np.float64)
    ref64 = np.asarray(ref64, dtype=np.float64)
    assert got.shape == ref64.shape, (got.shape, ref64.shape)
    if got.size == 0:
        return
    err = np.abs(got - ref64)
    bound = FP32_ATOL + FP32_RTOL * np.abs(ref64)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(int(np.argmax(np.where(bad, err / bound, 0))), got.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} fp32 outputs out of tolerance; worst at {idx}: "
            f"got {got[idx]!r}, want {ref64[idx]!r}")


def f16_ordinal(a: np.ndarray) -> np.ndarray:
    """Map binary16 values to integers that are monotonic in value (+0 == -0 == 0)."""
    b = np.ascontiguousarray(a, dtype=np.float16).view(np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def assert_f16_close(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    got = np.asarray(got, dtype=np.float16)
    want = np.asarray(want, dtype=np.float16)
    assert got.shape == want.shape, (got.shape, want.shape)
    if got.size == 0:
        return
    d = np.abs(f16_ordinal(got) - f16_ordinal(want))
    worst = int(d.max())
    if worst > F16_MAX_ULPS:
        idx = np.unravel_index(int(d.argmax()), d.shape)
        n_bad = int((d > F16_MAX_ULPS).sum())
        raise AssertionError(
            f"{what}: {n_bad} fp16 outputs beyond {F16_MAX_ULPS} ulp; worst {worst} ulp at "
            f"{idx}: got {got[idx]!r}, want {want[idx]!r}")


def assert_rounded_close(got: np.ndarray, want: np.ndarray, dtype: str, what: str = "") -> None:
    """16-bit storage: ``want`` is the oracle's result rounded once to ``dtype``."""
    if dtype == "bf16":
        assert_bf16_close(got, want, what)
    elif dtype == "f16":
        assert_f16_close(got, want, what)
    else:
        raise ValueError(f"not a 16-bit storage type: {dtype!r}")


def half_ulp(a: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of ``dtype`` at magnitude |a| (fp64 in, fp64 out)."""
    if dtype == "bf16":
        mant, emin = 8, -126
    elif dtype == "f16":
        mant, emin = 11, -14
    else:
        raise ValueError(f"not a 16-bit storage type: {dtype!r}")
    e = np.floor(np.log2(np.maximum(np.abs(a), 2.0 ** emin)))
    return np.ldexp(1.0, (e - mant).astype(np.int64))
