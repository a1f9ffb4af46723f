"""Pins for the CPU oracle: closed forms, invariants, library routines, brute force.

None of these checks re-types the oracle's own formula. Each one ties the oracle to
something fixed independently of it:

* bf16 rounding: hand-derived bit patterns at ties, overflow and subnormal boundaries,
  and torch's fp32 -> bf16 conversion (a library routine) on exactly representable input;
* fp16 (IEEE binary16) rounding: hand-derived bit patterns, numpy's float64 -> float16
  conversion (one rounding) and its float16 decoding of every pattern;
* RMSNorm (xserv "phase 4" design notes, RMSNorm section: y = x / sqrt(sum(x^2)/hidden
  + eps) * gamma): worked cases in exact closed form, the constant-row closed form,
  the zero row, positive-scale invariance and odd symmetry at eps = 0, numpy's vector
  norm, and exact rational arithmetic on tiny inputs;
* rotate-half RoPE (gollamago README "RoPE"; tilelang tutorial ch. 02, E13 pair
  formula): position 0 is the identity, the D = 2 worked case, per-pair norm
  preservation, composition of rotations, complex multiplication in numpy, and the
  interleaved pair formula on de-interleaved input;
* single rounding: a crafted case whose exact result rounds differently when rounded
  twice (fp64 -> fp32 -> bf16).
"""

from __future__ import annotations

import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

getcontext().prec = 50


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


# ------------------------------------------------------------------------ bf16 rounding

TWO = 2.0

BF16_HAND = [
    (1.0, 0x3F80),
    (-2.0, 0xC000),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (math.inf, 0x7F80),
    (-math.inf, 0xFF80),
    (1.0 + TWO**-8, 0x3F80),                  # tie, even neighbour is below
    (1.0 + 3 * TWO**-8, 0x3F82),              # tie, even neighbour is above
    (1.0 + TWO**-8 + TWO**-30, 0x3F81),       # just above a tie (fp32 would hide the 2^-30)
    (1.0 + TWO**-8 - TWO**-40, 0x3F80),       # just below a tie
    (-(1.0 + 3 * TWO**-8), 0xBF82),
    ((2 - TWO**-7) * TWO**127, 0x7F7F),       # largest finite bf16
    ((2 - TWO**-8) * TWO**127, 0x7F80),       # tie above it: odd mantissa, rounds to inf
    ((2 - TWO**-8 - TWO**-20) * TWO**127, 0x7F7F),
    (TWO**-133, 0x0001),                      # smallest subnormal
    (TWO**-134, 0x0000),                      # tie between 0 and it: even is 0
    (3 * TWO**-134, 0x0002),                  # tie between 1 and 2 ulps: even is 2
    (TWO**-126, 0x0080),                      # smallest normal
    (127.5 * TWO**-133, 0x0080),              # tie between 127 and 128 subnormal ulps
    (TWO**-140, 0x0000),
]


@pytest.mark.parametrize("value,bits", BF16_HAND)
def test_bf16_round_hand(lib, value, bits):
    assert lib.oracle_bf16_round(value) == bits


def test_bf16_round_nan(lib):
    b = lib.oracle_bf16_round(math.nan)
    assert (b & 0x7F80) == 0x7F80 and (b & 0x007F) != 0


def test_bf16_round_matches_torch_on_fp32_inputs(lib):
    # For values that are exact fp32 numbers a direct fp64 -> bf16 rounding must agree
    # with torch's fp32 -> bf16 round-to-nearest-even conversion.
    g = torch.Generator().manual_seed(1234)
    bits = torch.randint(0, 2**32, (20000,), generator=g, dtype=torch.int64)
    f = bits.to(torch.int32).view(torch.float32)
    f = f[torch.isfinite(f)]
    extra = torch.tensor([1.00390625, 1.01171875, 3.3895314e38, 1e-40, -7.5e-39, 65504.0,
                          0.1, -0.3, 1e-45], dtype=torch.float32)
    f = torch.cat([f, extra])
    want = f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(f.double().numpy(), lib=lib)
    np.testing.assert_array_equal(got, want)


def test_bf16_value_matches_torch_on_every_pattern(lib):
    pats = np.arange(65536, dtype=np.uint16)
    want = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.bf16_value(pats, lib=lib)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


# IEEE binary16: hand-derived patterns around ties, overflow and the subnormal range.
F16_HAND = [
    (1.0, 0x3C00),
    (-2.0, 0xC000),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (1.0 + TWO**-10, 0x3C01),
    (1.0 + TWO**-11, 0x3C00),                 # tie between 1 and 1 + 2^-10: even is 1
    (1.0 + 3 * TWO**-11, 0x3C02),             # tie between mantissas 1 and 2: even is 2
    (1.0 + TWO**-11 + TWO**-30, 0x3C01),      # just above the tie
    (65504.0, 0x7BFF),                        # largest finite
    (65519.99, 0x7BFF),
    (65520.0, 0x7C00),                        # tie above it: odd mantissa, rounds to inf
    (-1e6, 0xFC00),
    (TWO**-14, 0x0400),                       # smallest normal
    (TWO**-24, 0x0001),                       # smallest subnormal
    (TWO**-25, 0x0000),                       # tie between 0 and it: even is 0
    (3 * TWO**-25, 0x0002),                   # tie between 1 and 2 ulps: even is 2
    (1023.5 * TWO**-24, 0x0400),              # tie between the largest subnormal and 2^-14
    (0.1, 0x2E66),
    (-3.14159265358979, 0xC248),
]


@pytest.mark.parametrize("value,bits", F16_HAND)
def test_f16_round_hand(lib, value, bits):
    assert lib.oracle_f16_round(value) == bits


def test_f16_round_nan(lib):
    b = lib.oracle_f16_round(math.nan)
    assert (b & 0x7C00) == 0x7C00 and (b & 0x03FF) != 0


def test_f16_round_matches_numpy_on_fp64_inputs(lib):
    # numpy converts float64 to float16 in one rounding to nearest, ties to even.
    rng = np.random.default_rng(99)
    mags = np.exp(rng.uniform(np.log(2.0**-27), np.log(7e4), 30000))
    vals = mags * rng.choice([-1.0, 1.0], mags.size)
    grid = np.arange(-2048, 2048, dtype=np.float64)
    ties = np.concatenate([(grid + 0.5) * 2.0**-24, (1024 + grid[2048:] + 0.5) * 2.0**-10,
                           (1024 + grid[2048:] + 0.5) * 2.0**5])
    vals = np.concatenate([vals, ties, [65504.0, 65519.0, 65520.0, 65535.0]])
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    got = oracle.f16_round(vals, lib=lib)
    np.testing.assert_array_equal(got, want)


def test_f16_value_matches_numpy_on_every_pattern(lib):
    pats = np.arange(65536, dtype=np.uint16)
    want = pats.view(np.float16).astype(np.float64)
    got = oracle.f16_value(pats, lib=lib)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


# ------------------------------------------------------------------------ RMSNorm

def _dsqrt(q: Fraction) -> Decimal:
    return (Decimal(q.numerator) / Decimal(q.denominator)).sqrt()


def _exact_rmsnorm(x_row, w, eps) -> list[float]:
    """y_j = x_j / sqrt(sum x^2 / n + eps) * w_j in exact rationals and a 50-digit sqrt."""
    xs = [Fraction(float(v)) for v in x_row]
    n = len(xs)
    mean = sum(v * v for v in xs) / n + Fraction(float(eps))
    rms = _dsqrt(mean)
    out = []
    for v, wj in zip(xs, w):
        num = Decimal(v.numerator) / Decimal(v.denominator) * Decimal(Fraction(float(wj)).numerator) \
            / Decimal(Fraction(float(wj)).denominator)
        out.append(float(num / rms))
    return out


@pytest.mark.parametrize("x,w,want", [
    # sum 25, mean 12.5
    ([3.0, 4.0], [1.0, 1.0], [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]),
    # sum 30, mean 7.5
    ([1.0, 2.0, 3.0, 4.0], [1.0] * 4, [k / math.sqrt(7.5) for k in (1, 2, 3, 4)]),
    ([1.0, 1.0, 1.0, 1.0], [2.0] * 4, [2.0] * 4),
    # w scales each column independently
    ([1.0, -1.0, 1.0, -1.0], [0.5, 2.0, -3.0, 4.0], [0.5, -2.0, -3.0, -4.0]),
])
def test_rmsnorm_worked_cases(lib, x, w, want):
    y = oracle.rmsnorm_f64(np.array([x]), np.array(w), 0.0, lib=lib)[0]
    np.testing.assert_allclose(y, want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("c", [1.0, -2.0, 0.01, -3.5e-3, 7.0, 1e3, -1e-4])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 1e-5, 0.25])
@pytest.mark.parametrize("cols", [1, 2, 7, 64, 3000])
def test_rmsnorm_constant_row_closed_form(lib, c, eps, cols):
    # x_j = c for every j: mean(x^2) = c^2, so y_j = w_j * sign(c) / sqrt(1 + eps / c^2).
    w = np.linspace(-1.5, 2.5, cols)
    y = oracle.rmsnorm_f64(np.full((1, cols), c), w, eps, lib=lib)[0]
    want = w * math.copysign(1.0, c) / math.sqrt(1.0 + eps / (c * c))
    np.testing.assert_allclose(y, want, rtol=1e-14, atol=1e-300)


def test_rmsnorm_zero_row(lib):
    y = oracle.rmsnorm_f64(np.zeros((2, 33)), np.linspace(-2, 2, 33), 1e-5, lib=lib)
    assert np.all(y == 0.0)


@pytest.mark.parametrize("alpha", [2.0, 0.125, 3.7, 1e-3, 1e3, 1e150])
def test_rmsnorm_scale_invariance_and_odd_symmetry(lib, alpha):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((3, 129))
    w = 1 + 0.1 * rng.standard_normal(129)
    y = oracle.rmsnorm_f64(x, w, 0.0, lib=lib)
    ys = oracle.rmsnorm_f64(alpha * x, w, 0.0, lib=lib)
    np.testing.assert_allclose(ys, y, rtol=1e-14, atol=0)
    yn = oracle.rmsnorm_f64(-x, w, 0.0, lib=lib)
    np.testing.assert_array_equal(yn, -y)


def test_rmsnorm_matches_numpy_vector_norm(lib):
    # eps = 0: rms(x) = ||x||_2 / sqrt(n), with numpy's norm as the library routine.
    rng = np.random.default_rng(11)
    for n in (1, 5, 64, 2048, 3001):
        x = rng.standard_normal((2, n))
        w = rng.standard_normal(n)
        y = oracle.rmsnorm_f64(x, w, 0.0, lib=lib)
        for r in range(2):
            rms = np.linalg.norm(x[r]) / math.sqrt(n)
            np.testing.assert_allclose(y[r], x[r] * w / rms, rtol=1e-13, atol=0)


def test_rmsnorm_eps_enters_the_mean_not_the_sum(lib):
    # cols = 4, x = [1,1,1,1], eps = 1: rms = sqrt(1 + 1) (not sqrt((4 + 1) / 4)).
    y = oracle.rmsnorm_f64(np.ones((1, 4)), np.ones(4), 1.0, lib=lib)[0]
    np.testing.assert_allclose(y, [1 / math.sqrt(2.0)] * 4, rtol=1e-15)


def test_rmsnorm_brute_force_exact_rationals(lib):
    rng = np.random.default_rng(3)
    for rows in (1, 2, 3):
        for cols in range(1, 34):
            x = rng.standard_normal((rows, cols)) * rng.choice([1e-3, 1.0, 1e3])
            w = 1 + 0.1 * rng.standard_normal(cols)
            eps = float(rng.choice([0.0, 1e-6, 1e-5]))
            y = oracle.rmsnorm_f64(x, w, eps, lib=lib)
            for r in range(rows):
                want = _exact_rmsnorm(x[r], w, eps)
                np.testing.assert_allclose(y[r], want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_rmsnorm_storage_path_rounds_the_fp64_result_once(lib, dtype):
    rng = np.random.default_rng(5)
    xf = rng.standard_normal((7, 300)).astype(np.float32)
    wf = (1 + 0.1 * rng.standard_normal(300)).astype(np.float32)
    if dtype == "bf16":
        xs = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        ws = torch.from_numpy(wf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        xd = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).double().numpy()
        wd = torch.from_numpy(ws.view(np.int16)).view(torch.bfloat16).double().numpy()
    elif dtype == "f16":
        xs, ws = xf.astype(np.float16), wf.astype(np.float16)
        xd, wd = xs.astype(np.float64), ws.astype(np.float64)
    else:
        xs, ws, xd, wd = xf, wf, xf.astype(np.float64), wf.astype(np.float64)
    y = oracle.rmsnorm(xs, ws, 1e-5, dtype, lib=lib)
    exact = np.array([_exact_rmsnorm(xd[r], wd, 1e-5) for r in range(7)])
    if dtype == "bf16":
        # The exact values (to ~1e-16) rounded once by the hand-pinned bf16 rounding.
        want = oracle.bf16_round(exact, lib=lib)
        np.testing.assert_array_equal(y, want)
    elif dtype == "f16":
        np.testing.assert_array_equal(y, exact.astype(np.float16))   # numpy: one rounding
    else:
        np.testing.assert_array_equal(y, exact.astype(np.float32))


def test_rmsnorm_thread_split_does_not_change_results(lib):
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal((37, 513)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((1 + 0.1 * rng.standard_normal(513)).astype(np.float32)).to(torch.bfloat16)
    xs = x.view(torch.int16).numpy().view(np.uint16)
    ws = w.view(torch.int16).numpy().view(np.uint16)
    a = oracle.rmsnorm(xs, ws, 1e-5, "bf16", nthreads=1, lib=lib)
    b = oracle.rmsnorm(xs, ws, 1e-5, "bf16", nthreads=3, lib=lib)
    c = oracle.rmsnorm(xs, ws, 1e-5, "bf16", nthreads=0, lib=lib)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)


def test_rmsnorm_argument_checks(lib):
    with pytest.raises(ValueError):
        oracle.rmsnorm_f64(np.zeros((1, 0)), np.zeros(0), 1e-5, lib=lib)
    with pytest.raises(ValueError):
        oracle.rmsnorm_f64(np.zeros((1, 3)), np.zeros(3), -1.0, lib=lib)
    assert oracle.rmsnorm_f64(np.zeros((0, 3)), np.zeros(3), 1e-5, lib=lib).shape == (0, 3)


# ------------------------------------------------------------------------ residual add

def _storage_pair(rng, shape, dtype, scale=1.0):
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    t = torch.from_numpy(f)
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
        return t, t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "f16":
        t = t.to(torch.float16)
        return t, t.numpy()
    return t, f


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_add_rmsnorm_h_is_the_library_sum_and_y_the_rmsnorm_of_h(lib, dtype):
    # h must equal torch's storage-type addition (round to nearest even of the exact sum),
    # and y the (separately pinned) RMSNorm of h as stored.
    rng = np.random.default_rng(31)
    for scale_r in (1.0, 1e-3, 300.0):
        xt, xs = _storage_pair(rng, (7, 301), dtype)
        rt, rs = _storage_pair(rng, (7, 301), dtype, scale_r)
        wt, ws = _storage_pair(rng, (301,), dtype, 0.1)
        ws = (torch.from_numpy(np.ones(301, np.float32)).to(wt.dtype) + wt)
        ws = ws.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else ws.numpy()
        h, y = oracle.add_rmsnorm(xs, rs, ws, 1e-5, dtype, lib=lib)
        want_h = xt + rt
        want_h = (want_h.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16"
                  else want_h.numpy())
        if dtype == "f16":   # the library sum of two binary16 values, rounded once
            assert want_h.dtype == np.float16
        np.testing.assert_array_equal(h, want_h)
        np.testing.assert_array_equal(y, oracle.rmsnorm(h, ws, 1e-5, dtype, lib=lib))


def test_add_rmsnorm_zero_residual_is_rmsnorm(lib):
    rng = np.random.default_rng(32)
    _, xs = _storage_pair(rng, (5, 64), "bf16")
    _, ws = _storage_pair(rng, (64,), "bf16")
    zero = np.zeros_like(xs)
    h, y = oracle.add_rmsnorm(xs, zero, ws, 1e-5, "bf16", lib=lib)
    np.testing.assert_array_equal(h, xs)
    np.testing.assert_array_equal(y, oracle.rmsnorm(xs, ws, 1e-5, "bf16", lib=lib))


# ------------------------------------------------------------------------ KV norm + rope + cache

@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_kv_cache_scatter_is_rmsnorm_and_rope_of_each_token(lib, dtype):
    # Every written cache row must equal the (separately pinned) RMSNorm of the token's left
    # part and rotate-half RoPE of its right part with table row s; padding slots (negative
    # or past the end) and rows no token names stay as they were.
    rng = np.random.default_rng(41)
    B, S, Dn, Dr, nslots = 2, 5, 24, 8, 16
    kvt, kvs = _storage_pair(rng, (B, S, Dn + Dr), dtype)
    _, gs = _storage_pair(rng, (Dn,), dtype)
    sin_t = rng.uniform(-1, 1, (S, Dr // 2)).astype(np.float32)
    cos_t = rng.uniform(-1, 1, (S, Dr // 2)).astype(np.float32)
    slots = rng.permutation(nslots)[:B * S].astype(np.int64)
    slots[3] = -1
    slots[7] = nslots + 2
    _, cn0 = _storage_pair(rng, (nslots, Dn), dtype)
    _, cr0 = _storage_pair(rng, (nslots, Dr), dtype)
    cn, cr = oracle.kv_rmsnorm_rope_cache(kvs, gs, sin_t, cos_t, slots, cn0, cr0, Dn, 1e-5,
                                          dtype, lib=lib)
    written = set()
    for t in range(B * S):
        b, s_ = divmod(t, S)
        slot = int(slots[t])
        if not 0 <= slot < nslots:
            continue
        written.add(slot)
        tok = kvs[b, s_]
        want_n = oracle.rmsnorm(tok[None, :Dn], gs, 1e-5, dtype, lib=lib)[0]
        want_r = oracle.rope(tok[None, None, None, Dn:], sin_t[s_:s_ + 1], cos_t[s_:s_ + 1],
                             dtype, lib=lib)[0, 0, 0]
        np.testing.assert_array_equal(cn[slot], want_n)
        np.testing.assert_array_equal(cr[slot], want_r)
    for slot in set(range(nslots)) - written:
        np.testing.assert_array_equal(cn[slot], cn0[slot])
        np.testing.assert_array_equal(cr[slot], cr0[slot])


# ------------------------------------------------------------------------ KV cat + head repeat

@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("B,P,S,Hk,D,n_rep", [(2, 5, 3, 3, 8, 4), (1, 0, 4, 2, 6, 1),
                                               (1, 7, 0, 1, 4, 3), (3, 1, 1, 4, 2, 2)])
def test_kv_cat_repeat_without_tables_is_numpy_concatenate_and_repeat(lib, dtype, B, P, S, Hk,
                                                                      D, n_rep):
    rng = np.random.default_rng(71 + P)
    _, past = _storage_pair(rng, (B, P, Hk, D), dtype)
    _, new = _storage_pair(rng, (B, S, Hk, D), dtype)
    out = oracle.kv_cat_repeat(past if P else None, new, None, None, n_rep, dtype, lib=lib)
    want = np.repeat(np.concatenate([past, new], axis=1), n_rep, axis=2)
    np.testing.assert_array_equal(out, want)


def test_kv_cat_repeat_rotates_new_rows_at_their_absolute_positions(lib):
    # fp32 storage: the rotated rows are numpy's complex product (x1 + i x2)(c + i s) with the
    # table row P + s, rounded to fp32; past rows pass through untouched; every repeated
    # copy of a head is the same
    rng = np.random.default_rng(72)
    B, P, S, Hk, D, n_rep = 2, 6, 3, 3, 8, 4
    past = rng.standard_normal((B, P, Hk, D)).astype(np.float32)
    new = rng.standard_normal((B, S, Hk, D)).astype(np.float32)
    ang = rng.uniform(-4, 4, (P + S, D // 2))
    sin, cos = np.sin(ang).astype(np.float32), np.cos(ang).astype(np.float32)
    out = oracle.kv_cat_repeat(past, new, sin, cos, n_rep, "f32", lib=lib)
    o = out.reshape(B, P + S, Hk, n_rep, D)
    for r in range(1, n_rep):
        np.testing.assert_array_equal(o[:, :, :, r], o[:, :, :, 0])
    np.testing.assert_array_equal(o[:, :P, :, 0], past)
    half = D // 2
    z = (new[..., :half].astype(np.float64) + 1j * new[..., half:].astype(np.float64)) * \
        (cos[P:].astype(np.float64) + 1j * sin[P:].astype(np.float64))[None, :, None, :]
    want = np.concatenate([z.real, z.imag], axis=-1).astype(np.float32)
    np.testing.assert_allclose(o[:, P:, :, 0], want, rtol=2e-7, atol=1e-30)


def test_kv_cat_repeat_argument_errors(lib):
    new = np.zeros((1, 2, 1, 4), np.float32)
    t = np.zeros((2, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.kv_cat_repeat(None, new, t, None, 2, "f32", lib=lib)     # one table only
    with pytest.raises(ValueError):
        oracle.kv_cat_repeat(None, new, None, None, 0, "f32", lib=lib)  # n_rep < 1


# ------------------------------------------------------------------------ LayerNorm

def test_layernorm_worked_case(lib):
    # [1, 2, 3, 4]: mean 2.5, var 1.25 -> (x - 2.5) / sqrt(1.25); then gamma 2, beta -1.
    y, _ = oracle.layernorm_f64(np.array([[1.0, 2.0, 3.0, 4.0]]), np.full(4, 2.0),
                                np.full(4, -1.0), 0.0, lib=lib)
    want = [2 * (k - 2.5) / math.sqrt(1.25) - 1 for k in (1, 2, 3, 4)]
    np.testing.assert_allclose(y[0], want, rtol=1e-15)


def test_layernorm_constant_row_gives_beta(lib):
    # x_j = c: every deviation is 0, so y = beta exactly (eps > 0).
    b = np.linspace(-1, 1, 33)
    y, _ = oracle.layernorm_f64(np.full((2, 33), 7.25), np.linspace(0.5, 2, 33), b, 1e-5, lib=lib)
    np.testing.assert_array_equal(y, np.stack([b, b]))


@pytest.mark.parametrize("a,shift", [(2.0, 0.0), (0.01, 100.0), (1e3, -3.0)])
def test_layernorm_affine_invariance(lib, a, shift):
    # eps = 0: LayerNorm(a x + b) = LayerNorm(x) for a > 0.
    rng = np.random.default_rng(61)
    x = rng.standard_normal((3, 257))
    g, b = rng.standard_normal(257), rng.standard_normal(257)
    y1, _ = oracle.layernorm_f64(x, g, b, 0.0, lib=lib)
    y2, _ = oracle.layernorm_f64(a * x + shift, g, b, 0.0, lib=lib)
    np.testing.assert_allclose(y2, y1, rtol=1e-9, atol=1e-10)


def test_layernorm_matches_numpy_mean_and_std(lib):
    # numpy's mean and population std (ddof = 0) as the library routines.
    rng = np.random.default_rng(62)
    for n in (1, 2, 7, 768, 4099):
        x = rng.standard_normal((2, n)) * 3 + 50
        g, b = rng.standard_normal(n), rng.standard_normal(n)
        y, _ = oracle.layernorm_f64(x, g, b, 1e-5, lib=lib)
        for r in range(2):
            want = (x[r] - x[r].mean()) / np.sqrt(x[r].var() + 1e-5) * g + b
            np.testing.assert_allclose(y[r], want, rtol=1e-9, atol=1e-12)


def test_layernorm_brute_force_exact_rationals(lib):
    rng = np.random.default_rng(63)
    for cols in range(1, 20):
        x = rng.standard_normal(cols) * rng.choice([1e-3, 1.0, 1e3]) + rng.choice([0.0, 100.0])
        g, b = rng.standard_normal(cols), rng.standard_normal(cols)
        eps = float(rng.choice([1e-6, 1e-5, 0.5]))
        y, _ = oracle.layernorm_f64(x[None], g, b, eps, lib=lib)
        xs = [Fraction(float(v)) for v in x]
        mean = sum(xs) / cols
        var = sum((v - mean) ** 2 for v in xs) / cols + Fraction(eps)
        den = _dsqrt(var)
        # fp64 rounds the mean by ~u|mean|; relative to a deviation that is |mean| / sigma.
        cond = 1 + abs(float(mean)) / float(den)
        for j in range(cols):
            d = xs[j] - mean
            want = Decimal(d.numerator) / Decimal(d.denominator) / den * Decimal(float(g[j])) \
                + Decimal(float(b[j]))
            bound = 1e-14 * cond * (1 + abs(float(d / 1) / float(den) * float(g[j])) + abs(b[j]))
            assert abs(y[0, j] - float(want)) <= bound


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_layernorm_storage_path_rounds_the_fp64_result_once(lib, dtype):
    rng = np.random.default_rng(64)
    xt, xs = _storage_pair(rng, (5, 300), dtype)
    _, gs = _storage_pair(rng, (300,), dtype)
    _, bs = _storage_pair(rng, (300,), dtype, 0.1)
    dec = (lambda a: oracle.bf16_value(a, lib=lib)) if dtype == "bf16" else (lambda a: a.astype(np.float64))
    y64, _ = oracle.layernorm_f64(dec(xs), dec(gs), dec(bs), 1e-5, lib=lib)
    y = oracle.layernorm(xs, gs, bs, 1e-5, dtype, lib=lib)
    if dtype == "bf16":
        want = oracle.bf16_round(y64, lib=lib)
    elif dtype == "f16":
        want = y64.astype(np.float16)          # numpy: one rounding from fp64
    else:
        want = y64.astype(np.float32)
    np.testing.assert_array_equal(y, want)


# ------------------------------------------------------------------------ interleaved RoPE, tables

def _f32_ulps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_rope_interleaved_is_rotate_half_on_deinterleaved_input(lib, dtype):
    # Interleaved RoPE at positions p_t equals the (separately pinned) rotate-half RoPE of the
    # de-interleaved heads with the table rows p_t, re-interleaved; tokens with a position
    # outside the table are left as they were.
    rng = np.random.default_rng(51)
    T, H, D, P = 9, 3, 12, 20
    xt, xs = _storage_pair(rng, (T, H, D), dtype)
    _, y0 = _storage_pair(rng, (T, H, D), dtype)
    sin_t = rng.uniform(-1, 1, (P, D // 2)).astype(np.float32)
    cos_t = rng.uniform(-1, 1, (P, D // 2)).astype(np.float32)
    pos = rng.integers(0, P, T).astype(np.int32)
    pos[2] = -3
    pos[5] = P
    y = oracle.rope_interleaved(xs, sin_t, cos_t, pos, y0, dtype, lib=lib)
    for t in range(T):
        if not 0 <= pos[t] < P:
            np.testing.assert_array_equal(y[t], y0[t])
            continue
        half = np.concatenate([xs[t][:, 0::2], xs[t][:, 1::2]], axis=-1)     # [H, D]
        r = oracle.rope(half[None, None], sin_t[pos[t]:pos[t] + 1], cos_t[pos[t]:pos[t] + 1],
                        dtype, lib=lib)[0, 0]
        np.testing.assert_array_equal(y[t][:, 0::2], r[:, :D // 2])
        np.testing.assert_array_equal(y[t][:, 1::2], r[:, D // 2:])


def test_rope_tables_match_numpy_and_closed_forms(lib):
    P, D, theta = 4097, 128, 500000.0
    s, c = oracle.rope_tables(P, D, theta, lib=lib)
    np.testing.assert_array_equal(s[0], 0.0)                 # position 0: angle 0
    np.testing.assert_array_equal(c[0], 1.0)
    # column 0: theta^0 = 1, angle = p exactly
    p = np.arange(P, dtype=np.float64)
    assert _f32_ulps(s[:, 0], np.sin(p).astype(np.float32)).max() <= 1
    # everything: numpy's own fp64 pow / sin / cos (the benchmark's host recipe)
    from block_memory_bound_gb300 import inputs
    ns, nc = inputs.rope_tables(P, D, theta)
    assert _f32_ulps(s, ns).max() <= 1 and _f32_ulps(c, nc).max() <= 1
    # the two columns are a rotation: sin^2 + cos^2 = 1 up to fp32 rounding
    assert np.abs(s.astype(np.float64) ** 2 + c.astype(np.float64) ** 2 - 1).max() < 2e-7


# ------------------------------------------------------------------------ RoPE

def _tables(S, half, angle_fn, dtype=np.float64):
    ang = np.array([[angle_fn(s, i) for i in range(half)] for s in range(S)], dtype=np.float64)
    return np.sin(ang).astype(dtype), np.cos(ang).astype(dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [2, 8, 64, 128, 6])
def test_rope_position_zero_is_identity(lib, dtype, D):
    # cos = 1, sin = 0 at position 0: the rotation is the identity, exactly.
    rng = np.random.default_rng(D)
    xf = rng.standard_normal((2, 1, 3, D)).astype(np.float32)
    x = (torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
         if dtype == "bf16" else xf)
    sin_t = np.zeros((1, D // 2), np.float32)
    cos_t = np.ones((1, D // 2), np.float32)
    y = oracle.rope(x, sin_t, cos_t, dtype, lib=lib)
    np.testing.assert_array_equal(y, x)


def test_rope_worked_case_d2(lib):
    # D = 2, angle 1 rad: [1, 0] -> [cos 1, sin 1] and [0, 1] -> [-sin 1, cos 1].
    s1 = np.float32(math.sin(1.0))
    c1 = np.float32(math.cos(1.0))
    sin_t = np.array([[s1]], np.float32)
    cos_t = np.array([[c1]], np.float32)
    x = np.array([[[[1.0, 0.0], [0.0, 1.0]]]], np.float32)       # B=1, S=1, H=2, D=2
    y = oracle.rope(x, sin_t, cos_t, "f32", lib=lib)
    np.testing.assert_array_equal(y[0, 0, 0], [c1, s1])
    np.testing.assert_array_equal(y[0, 0, 1], [-s1, c1])
    # fp32 table values are within half an fp32 ulp (< 6e-8) of cos 1 and sin 1
    assert abs(float(c1) - 0.540302306) < 1e-7 and abs(float(s1) - 0.841470985) < 1e-7


def test_rope_preserves_pair_norms(lib):
    rng = np.random.default_rng(21)
    B, S, H, D = 2, 5, 3, 16
    x = rng.standard_normal((B, S, H, D))
    sin_t, cos_t = _tables(S, D // 2, lambda s, i: 0.37 * s + 0.11 * i, np.float32)
    y = oracle.rope_f64(x, sin_t, cos_t, lib=lib)
    h = D // 2
    c = cos_t.astype(np.float64)[None, :, None, :]
    s = sin_t.astype(np.float64)[None, :, None, :]
    lhs = y[..., :h] ** 2 + y[..., h:] ** 2
    rhs = (c * c + s * s) * (x[..., :h] ** 2 + x[..., h:] ** 2)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12)


def test_rope_composition_of_rotations(lib):
    rng = np.random.default_rng(4)
    B, S, H, D = 1, 4, 2, 12
    x = rng.standard_normal((B, S, H, D))
    sa, ca = _tables(S, D // 2, lambda s, i: 0.3 + 0.2 * s - 0.05 * i)
    sb, cb = _tables(S, D // 2, lambda s, i: -1.1 + 0.07 * s * i)
    sab, cab = _tables(S, D // 2, lambda s, i: (0.3 + 0.2 * s - 0.05 * i) + (-1.1 + 0.07 * s * i))
    two_step = oracle.rope_f64(oracle.rope_f64(x, sa, ca, lib=lib), sb, cb, lib=lib)
    one_step = oracle.rope_f64(x, sab, cab, lib=lib)
    np.testing.assert_allclose(two_step, one_step, rtol=0, atol=1e-12)


def test_rope_is_complex_multiplication(lib):
    # (x_i + j x_{i+D/2}) * (cos + j sin) with the table row of the sequence index s,
    # broadcast over batch and heads (numpy complex128 as the library routine).
    rng = np.random.default_rng(8)
    B, S, H, D = 3, 5, 4, 10
    h = D // 2
    x = rng.standard_normal((B, S, H, D))
    sin_t = rng.standard_normal((S, h)).astype(np.float32)
    cos_t = rng.standard_normal((S, h)).astype(np.float32)
    y = oracle.rope_f64(x, sin_t, cos_t, lib=lib)
    z = (x[..., :h] + 1j * x[..., h:]) * (cos_t.astype(np.float64) + 1j * sin_t.astype(np.float64))[None, :, None, :]
    np.testing.assert_allclose(y[..., :h], z.real, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(y[..., h:], z.imag, rtol=1e-14, atol=1e-14)


def test_rope_rotate_half_equals_interleaved_on_deinterleaved_input(lib):
    # Interleaved RoPE (xserv rope kernel: pairs (x[2i], x[2i+1]), y0 = x0 c - x1 s,
    # y1 = x0 s + x1 c), written out with plain loops on the interleaved layout.
    rng = np.random.default_rng(13)
    B, S, H, D = 2, 3, 2, 8
    h = D // 2
    x = rng.standard_normal((B, S, H, D))
    sin_t = rng.uniform(-1, 1, (S, h))
    cos_t = rng.uniform(-1, 1, (S, h))
    inter = np.empty_like(x)
    inter[..., 0::2] = x[..., :h]
    inter[..., 1::2] = x[..., h:]
    out = np.empty_like(inter)
    for b in range(B):
        for s in range(S):
            for hh in range(H):
                for i in range(h):
                    x0, x1 = inter[b, s, hh, 2 * i], inter[b, s, hh, 2 * i + 1]
                    c, sn = cos_t[s, i], sin_t[s, i]
                    out[b, s, hh, 2 * i] = x0 * c - x1 * sn
                    out[b, s, hh, 2 * i + 1] = x0 * sn + x1 * c
    y = oracle.rope_f64(x, sin_t, cos_t, lib=lib)
    np.testing.assert_allclose(y[..., :h], out[..., 0::2], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(y[..., h:], out[..., 1::2], rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_rope_storage_path_rounds_the_fp64_result_once(lib, dtype):
    rng = np.random.default_rng(17)
    B, S, H, D = 2, 6, 3, 32
    xf = rng.standard_normal((B, S, H, D)).astype(np.float32)
    sin_t = rng.uniform(-1, 1, (S, D // 2)).astype(np.float32)
    cos_t = rng.uniform(-1, 1, (S, D // 2)).astype(np.float32)
    if dtype == "bf16":
        xs = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        xd = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).double().numpy()
    elif dtype == "f16":
        xs = xf.astype(np.float16)
        xd = xs.astype(np.float64)
    else:
        xs, xd = xf, xf.astype(np.float64)
    y = oracle.rope(xs, sin_t, cos_t, dtype, lib=lib)
    # Products of a bf16/fp32 value and an fp32 value are exact in fp64, so the complex
    # product below is the exact result up to one fp64 rounding of each sum.
    z = (xd[..., :D // 2] + 1j * xd[..., D // 2:]) * (cos_t + 1j * sin_t.astype(np.float64))[None, :, None, :]
    exact = np.concatenate([z.real, z.imag], axis=-1)
    if dtype == "bf16":
        np.testing.assert_array_equal(y, oracle.bf16_round(exact, lib=lib))
    elif dtype == "f16":
        np.testing.assert_array_equal(y, exact.astype(np.float16))
    else:
        np.testing.assert_array_equal(y, exact.astype(np.float32))


def test_rope_single_rounding_crafted_case(lib):
    # y_0 = x_0 c - x_1 s = 1 * (1 + 2^-8) - 2^-10 * (-2^-20) = 1 + 2^-8 + 2^-30 exactly.
    # Rounded once to bf16 that is 0x3F81; rounded first to fp32 (1 + 2^-8, a tie) and
    # then to bf16 it would be 0x3F80.
    c = np.float32(1 + 2.0**-8)
    s = np.float32(-(2.0**-20))
    x = torch.tensor([[[[1.0, 2.0**-10]]]], dtype=torch.float32).to(torch.bfloat16)
    xs = x.view(torch.int16).numpy().view(np.uint16)
    y = oracle.rope(xs, np.array([[s]]), np.array([[c]]), "bf16", lib=lib)
    assert int(y[0, 0, 0, 0]) == 0x3F81


def test_rope_thread_split_does_not_change_results(lib):
    rng = np.random.default_rng(23)
    xf = rng.standard_normal((2, 9, 4, 64)).astype(np.float32)
    sin_t = rng.uniform(-1, 1, (9, 32)).astype(np.float32)
    cos_t = rng.uniform(-1, 1, (9, 32)).astype(np.float32)
    a = oracle.rope(xf, sin_t, cos_t, "f32", nthreads=1, lib=lib)
    b = oracle.rope(xf, sin_t, cos_t, "f32", nthreads=5, lib=lib)
    np.testing.assert_array_equal(a, b)


def test_rope_argument_checks(lib):
    with pytest.raises(ValueError):
        oracle.rope_f64(np.zeros((1, 1, 1, 3)), np.zeros((1, 1)), np.zeros((1, 1)), lib=lib)
    assert oracle.rope_f64(np.zeros((0, 2, 1, 4)), np.zeros((2, 2)), np.zeros((2, 2)),
                           lib=lib).shape == (0, 2, 1, 4)
