"""CPU oracle for RMSNorm forward and rotate-half RoPE (fp64, plain C++).

TEST INFRASTRUCTURE ONLY: the tests, the package entry point's smoke check and the
benchmark's CPU-baseline leg are the only callers. The product path (the CUDA library
and its Python binding) never imports this module, and this module never imports the
product package.

The arithmetic lives in ``camp_oracle.cpp`` (see its header for the definitions and the
passages they follow). This file only compiles that source with the host C++ compiler
and marshals numpy arrays through ctypes. bf16 arrays are passed as ``numpy.uint16`` bit
patterns, fp16 arrays as ``numpy.float16``, fp32 arrays as ``numpy.float32``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "camp_oracle.cpp")
LIBRARY = os.path.join(_HERE, "libcamp_oracle.so")

# Storage-type codes understood by the oracle's C entry points.
F16 = 0
F32 = 1
BF16 = 3

# -ffp-contract=off: no fused multiply-add may change a result between x86-64 and aarch64.
CXXFLAGS = ["-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def build(source: str = SOURCE, output: str = LIBRARY, force: bool = False) -> str:
    """Compile the oracle into a shared library (skipped when it is up to date)."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    cxx = os.environ.get("CXX", "g++")
    tmp = output + f".tmp{os.getpid()}"
    subprocess.run([cxx, *CXXFLAGS, source, "-o", tmp], check=True)
    os.replace(tmp, output)
    return output


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    i64, vp, dbl, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
    lib.oracle_bf16_round.argtypes = [dbl]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_value.restype = dbl
    lib.oracle_f16_round.argtypes = [dbl]
    lib.oracle_f16_round.restype = ctypes.c_uint16
    lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_value.restype = dbl
    lib.oracle_threads_available.argtypes = []
    lib.oracle_threads_available.restype = c_int
    lib.oracle_rmsnorm_f64.argtypes = [vp, vp, vp, i64, i64, dbl]
    lib.oracle_rmsnorm_f64.restype = c_int
    lib.oracle_rmsnorm.argtypes = [vp, vp, vp, i64, i64, dbl, c_int, c_int]
    lib.oracle_rmsnorm.restype = c_int
    lib.oracle_add_rmsnorm.argtypes = [vp, vp, vp, vp, vp, i64, i64, dbl, c_int, c_int]
    lib.oracle_add_rmsnorm.restype = c_int
    lib.oracle_kv_rmsnorm_rope_cache.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                                 i64, i64, dbl, c_int]
    lib.oracle_kv_rmsnorm_rope_cache.restype = c_int
    lib.oracle_layernorm_f64.argtypes = [vp, vp, vp, vp, vp, i64, i64, dbl]
    lib.oracle_layernorm_f64.restype = c_int
    lib.oracle_layernorm.argtypes = [vp, vp, vp, vp, i64, i64, dbl, c_int, c_int]
    lib.oracle_layernorm.restype = c_int
    lib.oracle_kv_cat_repeat.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int]
    lib.oracle_kv_cat_repeat.restype = c_int
    lib.oracle_rope_interleaved.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, c_int]
    lib.oracle_rope_interleaved.restype = c_int
    lib.oracle_rope_tables.argtypes = [vp, vp, i64, i64, dbl]
    lib.oracle_rope_tables.restype = c_int
    lib.oracle_rope_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64]
    lib.oracle_rope_f64.restype = c_int
    lib.oracle_rope.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, c_int, c_int]
    lib.oracle_rope.restype = c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Build (if needed) and load the oracle library. ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _storage(dtype: str) -> tuple[int, type]:
    if dtype == "bf16":
        return BF16, np.uint16
    if dtype == "f32":
        return F32, np.float32
    if dtype == "f16":
        return F16, np.float16
    raise ValueError(f"unknown storage type {dtype!r}")


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"{what}: oracle returned status {rc}")


def threads_available(lib: ctypes.CDLL | None = None) -> int:
    return (lib or load()).oracle_threads_available()


def bf16_round(values, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """fp64 values -> bf16 bit patterns, rounded once to nearest, ties to even."""
    lib = lib or load()
    v = np.asarray(values, dtype=np.float64).ravel()
    out = np.fromiter((lib.oracle_bf16_round(float(t)) for t in v), dtype=np.uint16,
                      count=v.size)
    return out.reshape(np.shape(values))


def bf16_value(bits, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """bf16 bit patterns -> their exact values as fp64."""
    lib = lib or load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.fromiter((lib.oracle_bf16_value(int(t)) for t in b), dtype=np.float64,
                      count=b.size)
    return out.reshape(np.shape(bits))


def f16_round(values, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """fp64 values -> IEEE binary16 bit patterns, rounded once to nearest, ties to even."""
    lib = lib or load()
    v = np.asarray(values, dtype=np.float64).ravel()
    out = np.fromiter((lib.oracle_f16_round(float(t)) for t in v), dtype=np.uint16,
                      count=v.size)
    return out.reshape(np.shape(values))


def f16_value(bits, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """binary16 bit patterns -> their exact values as fp64."""
    lib = lib or load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.fromiter((lib.oracle_f16_value(int(t)) for t in b), dtype=np.float64,
                      count=b.size)
    return out.reshape(np.shape(bits))


def rmsnorm_f64(x, w, eps: float, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Unrounded fp64 RMSNorm of fp64 ``x[rows, cols]`` with weight ``w[cols]``."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    rows, cols = x.shape
    assert w.shape == (cols,)
    y = np.empty_like(x)
    _check(lib.oracle_rmsnorm_f64(_ptr(x), _ptr(w), _ptr(y), rows, cols, float(eps)),
           "rmsnorm_f64")
    return y


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float, dtype: str, nthreads: int = 0,
            lib: ctypes.CDLL | None = None) -> np.ndarray:
    """RMSNorm of storage-typed ``x[rows, cols]``, ``w[cols]``: fp64 inside, one rounding."""
    lib = lib or load()
    code, npt = _storage(dtype)
    x = np.ascontiguousarray(x)
    w = np.ascontiguousarray(w)
    assert x.dtype == npt and w.dtype == npt, (x.dtype, w.dtype, dtype)
    rows, cols = x.shape
    assert w.shape == (cols,)
    y = np.empty_like(x)
    _check(lib.oracle_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, cols, float(eps), code,
                              int(nthreads)), "rmsnorm")
    return y


def add_rmsnorm(x: np.ndarray, r: np.ndarray, w: np.ndarray, eps: float, dtype: str,
                nthreads: int = 0, lib: ctypes.CDLL | None = None
                ) -> tuple[np.ndarray, np.ndarray]:
    """(h, y): h = x + r rounded once, y = RMSNorm(h as stored) * w rounded once."""
    lib = lib or load()
    code, npt = _storage(dtype)
    x = np.ascontiguousarray(x)
    r = np.ascontiguousarray(r)
    w = np.ascontiguousarray(w)
    assert x.dtype == npt and r.dtype == npt and w.dtype == npt
    assert r.shape == x.shape
    rows, cols = x.shape
    assert w.shape == (cols,)
    h = np.empty_like(x)
    y = np.empty_like(x)
    _check(lib.oracle_add_rmsnorm(_ptr(x), _ptr(r), _ptr(w), _ptr(h), _ptr(y), rows, cols,
                                  float(eps), code, int(nthreads)), "add_rmsnorm")
    return h, y


def kv_rmsnorm_rope_cache(kv: np.ndarray, gamma: np.ndarray, sin_t: np.ndarray,
                          cos_t: np.ndarray, slots: np.ndarray, cache_n: np.ndarray,
                          cache_r: np.ndarray, Dn: int, eps: float, dtype: str,
                          lib: ctypes.CDLL | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Copies of (cache_n, cache_r) after scattering RMSNorm(kv[..., :Dn]) * gamma and the
    rotate-half RoPE of kv[..., Dn:] of every token to the row its slot names."""
    lib = lib or load()
    code, npt = _storage(dtype)
    kv = np.ascontiguousarray(kv)
    B, S, W = kv.shape
    Dr = W - Dn
    gamma = np.ascontiguousarray(gamma)
    sin_t = np.ascontiguousarray(sin_t, dtype=np.float32)
    cos_t = np.ascontiguousarray(cos_t, dtype=np.float32)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    cn = np.array(cache_n, copy=True, order="C")
    cr = np.array(cache_r, copy=True, order="C")
    assert kv.dtype == npt and gamma.dtype == npt and cn.dtype == npt and cr.dtype == npt
    assert gamma.shape == (Dn,) and slots.shape == (B * S,)
    assert sin_t.shape == (S, Dr // 2) and cos_t.shape == (S, Dr // 2)
    assert cn.shape[1] == Dn and cr.shape[1] == Dr and cn.shape[0] == cr.shape[0]
    _check(lib.oracle_kv_rmsnorm_rope_cache(
        _ptr(kv), _ptr(gamma), _ptr(sin_t), _ptr(cos_t), _ptr(slots), _ptr(cn), _ptr(cr),
        B, S, Dn, Dr, cn.shape[0], float(eps), code), "kv_rmsnorm_rope_cache")
    return cn, cr


def layernorm_f64(x, gamma, beta, eps: float, lib: ctypes.CDLL | None = None
                  ) -> tuple[np.ndarray, np.ndarray]:
    """(y, scale): unrounded fp64 LayerNorm of fp64 x [rows, cols] and, per element,
    |xhat * gamma| + |beta| (the magnitude fp32 arithmetic errors are relative to)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(gamma, dtype=np.float64)
    b = np.ascontiguousarray(beta, dtype=np.float64)
    rows, cols = x.shape
    y = np.empty_like(x)
    scale = np.empty_like(x)
    _check(lib.oracle_layernorm_f64(_ptr(x), _ptr(g), _ptr(b), _ptr(y), _ptr(scale), rows, cols,
                                    float(eps)), "layernorm_f64")
    return y, scale


def layernorm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float, dtype: str,
              nthreads: int = 0, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """LayerNorm of storage-typed x [rows, cols]: fp64 inside, one rounding."""
    lib = lib or load()
    code, npt = _storage(dtype)
    x = np.ascontiguousarray(x)
    gamma = np.ascontiguousarray(gamma)
    beta = np.ascontiguousarray(beta)
    assert x.dtype == npt and gamma.dtype == npt and beta.dtype == npt
    rows, cols = x.shape
    y = np.empty_like(x)
    _check(lib.oracle_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), rows, cols,
                                float(eps), code, int(nthreads)), "layernorm")
    return y


def kv_cat_repeat(past, new, sin, cos, n_rep: int, dtype: str,
                  lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Storage-typed past [B, P, Hk, D] (or None when P = 0) and new [B, S, Hk, D] ->
    out [B, P+S, Hk*n_rep, D]: concatenated along the sequence, each head repeated n_rep
    times in place, new rows rotated at positions P + s with fp32 tables [P+S, D/2]
    (sin = cos = None: copied)."""
    lib = lib or load()
    code, npt = _storage(dtype)
    new = np.ascontiguousarray(new)
    assert new.dtype == npt and new.ndim == 4
    B, S, Hk, D = new.shape
    if past is None:
        past = np.zeros((B, 0, Hk, D), dtype=npt)
    past = np.ascontiguousarray(past)
    assert past.dtype == npt and past.shape[0] == B and past.shape[2:] == (Hk, D)
    P = past.shape[1]
    out = np.empty((B, P + S, Hk * max(int(n_rep), 0), D), dtype=npt)
    if sin is not None:
        sin = np.ascontiguousarray(sin, dtype=np.float32)
        assert sin.shape == (P + S, D // 2)
    if cos is not None:
        cos = np.ascontiguousarray(cos, dtype=np.float32)
        assert cos.shape == (P + S, D // 2)
    _check(lib.oracle_kv_cat_repeat(_ptr(past) if P else None, _ptr(new) if S else None,
                                    None if sin is None else _ptr(sin),
                                    None if cos is None else _ptr(cos), _ptr(out), B, P, S,
                                    Hk, D, int(n_rep), code), "kv_cat_repeat")
    return out


def rope_interleaved(x: np.ndarray, sin_t: np.ndarray, cos_t: np.ndarray,
                     positions: np.ndarray, y0: np.ndarray, dtype: str,
                     lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Interleaved RoPE of x [tokens, H, D] at table rows positions[t]; a copy of y0 with the
    rows of every token that has a valid position overwritten."""
    lib = lib or load()
    code, npt = _storage(dtype)
    x = np.ascontiguousarray(x)
    tokens, H, D = x.shape
    sin_t = np.ascontiguousarray(sin_t, dtype=np.float32)
    cos_t = np.ascontiguousarray(cos_t, dtype=np.float32)
    positions = np.ascontiguousarray(positions, dtype=np.int32)
    y = np.array(y0, copy=True, order="C")
    assert x.dtype == npt and y.dtype == npt and y.shape == x.shape
    assert sin_t.shape == cos_t.shape and sin_t.shape[1] == D // 2
    assert positions.shape == (tokens,)
    _check(lib.oracle_rope_interleaved(_ptr(x), _ptr(sin_t), _ptr(cos_t), _ptr(positions),
                                       _ptr(y), tokens, H, D, sin_t.shape[0], code),
           "rope_interleaved")
    return y


def rope_tables(max_pos: int, D: int, theta: float, lib: ctypes.CDLL | None = None
                ) -> tuple[np.ndarray, np.ndarray]:
    """(sin, cos) fp32 [max_pos, D/2]: angle = p * theta^(-2i/D) in fp64, rounded once."""
    lib = lib or load()
    sin_t = np.empty((max_pos, D // 2), np.float32)
    cos_t = np.empty((max_pos, D // 2), np.float32)
    _check(lib.oracle_rope_tables(_ptr(sin_t), _ptr(cos_t), max_pos, D, float(theta)),
           "rope_tables")
    return sin_t, cos_t


def rope_f64(x, sin_t, cos_t, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Unrounded fp64 rotate-half RoPE of ``x[B, S, H, D]`` with tables ``[S, D/2]``."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    sin_t = np.ascontiguousarray(sin_t, dtype=np.float64)
    cos_t = np.ascontiguousarray(cos_t, dtype=np.float64)
    B, S, H, D = x.shape
    assert sin_t.shape == (S, D // 2) and cos_t.shape == (S, D // 2)
    y = np.empty_like(x)
    _check(lib.oracle_rope_f64(_ptr(x), _ptr(sin_t), _ptr(cos_t), _ptr(y), B, S, H, D),
           "rope_f64")
    return y


def rope(x: np.ndarray, sin_t: np.ndarray, cos_t: np.ndarray, dtype: str,
         nthreads: int = 0, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Rotate-half RoPE of storage-typed ``x[B, S, H, D]`` with fp32 tables ``[S, D/2]``."""
    lib = lib or load()
    code, npt = _storage(dtype)
    x = np.ascontiguousarray(x)
    sin_t = np.ascontiguousarray(sin_t, dtype=np.float32)
    cos_t = np.ascontiguousarray(cos_t, dtype=np.float32)
    assert x.dtype == npt
    B, S, H, D = x.shape
    assert sin_t.shape == (S, D // 2) and cos_t.shape == (S, D // 2)
    y = np.empty_like(x)
    _check(lib.oracle_rope(_ptr(x), _ptr(sin_t), _ptr(cos_t), _ptr(y), B, S, H, D, code,
                           int(nthreads)), "rope")
    return y
