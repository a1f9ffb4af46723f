"""Python binding of libcamp's C ABI (``include/camp.h``): argument marshalling only.

The functions named like the C entry points (``camp_rmsnorm``, ``camp_rope``, ...) take
raw device pointers (ints) or torch tensors (their ``data_ptr()`` is passed), a dtype as
``camp.BF16``/``camp.F16``/``camp.F32`` or ``"bf16"``/``"f16"``/``"f32"``, and a stream as an int handle, a
``torch.cuda.Stream`` or ``None`` (torch's current stream on the current device). They
raise :class:`CampError` on any non-success status. Every step of the computation runs
in libcamp's kernels; there is no other code path. The library is opened on first use
and a missing library is an error, not a fallback.

:func:`rmsnorm` and :func:`rope` are tensor-level conveniences on top: they check
shapes, allocate the output with torch when none is given, and call the entry points.
"""

from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "libcamp.so")

SUCCESS = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED_DTYPE = 2
ERR_RUNTIME = 3
ERR_NOT_SUPPORTED = 5

F16 = 0
F32 = 1
BF16 = 3

KERNEL_RMSNORM_ROWS = 1
KERNEL_RMSNORM_WIDE = 2
KERNEL_ROPE = 3
KERNEL_ROPE_FLAT = 4
KERNEL_ROPE_SPLIT = 5
KERNEL_RMSNORM_CLUSTER = 6
KERNEL_KV_CACHE = 7
KERNEL_ROPE_INTERLEAVED = 8
KERNEL_LAYERNORM_ROWS = 9
KERNEL_KV_CAT = 10
KERNEL_RMSNORM_STAGED = 11
KERNEL_LAYERNORM_STAGED = 12
KERNEL_LAYERNORM_WIDE = 13
KERNEL_RMSNORM_SPREAD = 14
KERNEL_LAYERNORM_SPREAD = 15

DEVICE_ERROR_WAIT_TIMEOUT = 1

# Every symbol include/camp.h declares.
EXPORTS = (
    "camp_rmsnorm", "camp_rope", "camp_status_string", "camp_last_cuda_error",
    "camp_rmsnorm_plan", "camp_rope_plan", "camp_rmsnorm_with_plan", "camp_rope_with_plan",
    "camp_rope_qk", "camp_rope_qk_plan", "camp_rope_qk_with_plan",
    "camp_add_rmsnorm", "camp_add_rmsnorm_plan", "camp_add_rmsnorm_with_plan",
    "camp_kv_rmsnorm_rope_cache", "camp_kv_rmsnorm_rope_cache_plan",
    "camp_kv_rmsnorm_rope_cache_with_plan",
    "camp_rope_interleaved", "camp_rope_interleaved_plan", "camp_rope_interleaved_with_plan",
    "camp_rope_tables",
    "camp_layernorm", "camp_layernorm_plan", "camp_layernorm_with_plan",
    "camp_kv_cat_repeat", "camp_kv_cat_repeat_plan", "camp_kv_cat_repeat_with_plan",
    "camp_device_errors", "camp_layernorm_wait_probe", "camp_rmsnorm_wait_probe",
)


class CampError(RuntimeError):
    """A non-success status from libcamp."""

    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        msg = f"{fn}: {status_string(status)} (status {status})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


class Plan(ctypes.Structure):
    """Mirror of ``camp_plan_t``."""
    _fields_ = [
        ("kernel", ctypes.c_int32),
        ("vec_bytes", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("per_thread", ctypes.c_int32),
        ("block", ctypes.c_int32),
        ("cluster", ctypes.c_int32),
        ("grid", ctypes.c_int64),
        ("rows_per_step", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}

    def __repr__(self) -> str:
        return f"Plan({self.as_dict()})"


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


def load(path: str = LIBRARY) -> ctypes.CDLL:
    """Open libcamp.so (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libcamp.so is not built ({path}); run "
                "`python -m block_memory_bound_gb300.build` or __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i64, f32, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
        pplan = ctypes.POINTER(Plan)
        lib.camp_rmsnorm.argtypes = [vp, vp, vp, i64, i64, f32, c_int, vp]
        lib.camp_rmsnorm.restype = c_int
        lib.camp_rope.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, c_int, vp]
        lib.camp_rope.restype = c_int
        lib.camp_status_string.argtypes = [c_int]
        lib.camp_status_string.restype = ctypes.c_char_p
        lib.camp_last_cuda_error.argtypes = []
        lib.camp_last_cuda_error.restype = c_int
        lib.camp_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), c_int]
        lib.camp_device_errors.restype = c_int
        lib.camp_layernorm_wait_probe.argtypes = [vp, vp, vp, vp, i64, i64, f32, c_int, pplan,
                                                  ctypes.c_uint64, vp]
        lib.camp_layernorm_wait_probe.restype = c_int
        lib.camp_rmsnorm_wait_probe.argtypes = [vp, vp, vp, i64, i64, f32, c_int, pplan,
                                                ctypes.c_uint64, vp]
        lib.camp_rmsnorm_wait_probe.restype = c_int
        lib.camp_rmsnorm_plan.argtypes = [vp, vp, vp, i64, i64, c_int, pplan]
        lib.camp_rmsnorm_plan.restype = c_int
        lib.camp_rope_plan.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, c_int, pplan]
        lib.camp_rope_plan.restype = c_int
        lib.camp_rmsnorm_with_plan.argtypes = [vp, vp, vp, i64, i64, f32, c_int, pplan, vp]
        lib.camp_rmsnorm_with_plan.restype = c_int
        lib.camp_rope_with_plan.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, c_int, pplan, vp]
        lib.camp_rope_with_plan.restype = c_int
        lib.camp_add_rmsnorm.argtypes = [vp, vp, vp, vp, vp, i64, i64, f32, c_int, vp]
        lib.camp_add_rmsnorm.restype = c_int
        lib.camp_add_rmsnorm_plan.argtypes = [vp, vp, vp, vp, vp, i64, i64, c_int, pplan]
        lib.camp_add_rmsnorm_plan.restype = c_int
        lib.camp_add_rmsnorm_with_plan.argtypes = [vp, vp, vp, vp, vp, i64, i64, f32, c_int,
                                                   pplan, vp]
        lib.camp_add_rmsnorm_with_plan.restype = c_int
        lib.camp_layernorm.argtypes = [vp, vp, vp, vp, i64, i64, f32, c_int, vp]
        lib.camp_layernorm.restype = c_int
        lib.camp_layernorm_plan.argtypes = [vp, vp, vp, vp, i64, i64, c_int, pplan]
        lib.camp_layernorm_plan.restype = c_int
        lib.camp_layernorm_with_plan.argtypes = [vp, vp, vp, vp, i64, i64, f32, c_int, pplan, vp]
        lib.camp_layernorm_with_plan.restype = c_int
        ilsig = [vp, vp, vp, vp, vp, i64, i64, i64, i64, c_int]
        lib.camp_rope_interleaved.argtypes = ilsig + [vp]
        lib.camp_rope_interleaved.restype = c_int
        lib.camp_rope_interleaved_plan.argtypes = ilsig + [pplan]
        lib.camp_rope_interleaved_plan.restype = c_int
        lib.camp_rope_interleaved_with_plan.argtypes = ilsig + [pplan, vp]
        lib.camp_rope_interleaved_with_plan.restype = c_int
        lib.camp_rope_tables.argtypes = [vp, vp, i64, i64, ctypes.c_double, vp]
        lib.camp_rope_tables.restype = c_int
        kvsig = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64]
        lib.camp_kv_rmsnorm_rope_cache.argtypes = kvsig + [f32, c_int, vp]
        lib.camp_kv_rmsnorm_rope_cache.restype = c_int
        lib.camp_kv_rmsnorm_rope_cache_plan.argtypes = kvsig + [c_int, pplan]
        lib.camp_kv_rmsnorm_rope_cache_plan.restype = c_int
        lib.camp_kv_rmsnorm_rope_cache_with_plan.argtypes = kvsig + [f32, c_int, pplan, vp]
        lib.camp_kv_rmsnorm_rope_cache_with_plan.restype = c_int
        catsig = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int]
        lib.camp_kv_cat_repeat.argtypes = catsig + [vp]
        lib.camp_kv_cat_repeat.restype = c_int
        lib.camp_kv_cat_repeat_plan.argtypes = catsig + [pplan]
        lib.camp_kv_cat_repeat_plan.restype = c_int
        lib.camp_kv_cat_repeat_with_plan.argtypes = catsig + [pplan, vp]
        lib.camp_kv_cat_repeat_with_plan.restype = c_int
        qk = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int]
        lib.camp_rope_qk.argtypes = qk + [vp]
        lib.camp_rope_qk.restype = c_int
        lib.camp_rope_qk_plan.argtypes = qk + [pplan]
        lib.camp_rope_qk_plan.restype = c_int
        lib.camp_rope_qk_with_plan.argtypes = qk + [pplan, vp]
        lib.camp_rope_qk_with_plan.restype = c_int
        _lib = lib
        return lib


# ------------------------------------------------------------------ marshalling

def _ptr(a) -> int | None:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()   # torch.Tensor


def _dtype(d) -> int:
    if isinstance(d, int) and d in (F16, F32, BF16):
        return d
    if d in ("bf16", "bfloat16"):
        return BF16
    if d in ("f16", "fp16", "float16"):
        return F16
    if d in ("f32", "fp32", "float32"):
        return F32
    name = str(d)
    if name == "torch.bfloat16":
        return BF16
    if name == "torch.float16":
        return F16
    if name == "torch.float32":
        return F32
    if isinstance(d, int):
        return d   # passed through; the library rejects unknown codes
    raise ValueError(f"unknown dtype {d!r}")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream   # torch.cuda.Stream


def _check(fn: str, status: int) -> None:
    if status != SUCCESS:
        detail = ""
        if status == ERR_RUNTIME:
            detail = f"cudaError {load().camp_last_cuda_error()}"
        raise CampError(fn, status, detail)


# ------------------------------------------------------------------ C entry points

def status_string(status: int) -> str:
    return load().camp_status_string(int(status)).decode()


camp_status_string = status_string


def camp_last_cuda_error() -> int:
    return load().camp_last_cuda_error()


def camp_device_errors(clear: bool = False) -> int:
    """The library's device error word (0: no kernel's bounded wait ran out); synchronizes."""
    v = ctypes.c_uint32(0)
    _check("camp_device_errors", load().camp_device_errors(ctypes.byref(v), int(bool(clear))))
    return v.value


def camp_rmsnorm(x, w, y, rows: int, cols: int, eps: float, dtype, stream=None) -> None:
    _check("camp_rmsnorm", load().camp_rmsnorm(
        _ptr(x), _ptr(w), _ptr(y), int(rows), int(cols), float(eps), _dtype(dtype),
        _stream(stream)))


def camp_rope(x, sin, cos, y, B: int, S: int, H: int, D: int, dtype, stream=None) -> None:
    _check("camp_rope", load().camp_rope(
        _ptr(x), _ptr(sin), _ptr(cos), _ptr(y), int(B), int(S), int(H), int(D),
        _dtype(dtype), _stream(stream)))


def camp_rmsnorm_plan(x, w, y, rows: int, cols: int, dtype) -> Plan:
    p = Plan()
    _check("camp_rmsnorm_plan", load().camp_rmsnorm_plan(
        _ptr(x), _ptr(w), _ptr(y), int(rows), int(cols), _dtype(dtype), ctypes.byref(p)))
    return p


def camp_rope_plan(x, sin, cos, y, B: int, S: int, H: int, D: int, dtype) -> Plan:
    p = Plan()
    _check("camp_rope_plan", load().camp_rope_plan(
        _ptr(x), _ptr(sin), _ptr(cos), _ptr(y), int(B), int(S), int(H), int(D),
        _dtype(dtype), ctypes.byref(p)))
    return p


def camp_rmsnorm_with_plan(x, w, y, rows: int, cols: int, eps: float, dtype, plan: Plan,
                           stream=None) -> None:
    _check("camp_rmsnorm_with_plan", load().camp_rmsnorm_with_plan(
        _ptr(x), _ptr(w), _ptr(y), int(rows), int(cols), float(eps), _dtype(dtype),
        ctypes.byref(plan), _stream(stream)))


def camp_rope_with_plan(x, sin, cos, y, B: int, S: int, H: int, D: int, dtype, plan: Plan,
                        stream=None) -> None:
    _check("camp_rope_with_plan", load().camp_rope_with_plan(
        _ptr(x), _ptr(sin), _ptr(cos), _ptr(y), int(B), int(S), int(H), int(D),
        _dtype(dtype), ctypes.byref(plan), _stream(stream)))


def camp_add_rmsnorm(x, r, w, h, y, rows: int, cols: int, eps: float, dtype, stream=None) -> None:
    _check("camp_add_rmsnorm", load().camp_add_rmsnorm(
        _ptr(x), _ptr(r), _ptr(w), _ptr(h), _ptr(y), int(rows), int(cols), float(eps),
        _dtype(dtype), _stream(stream)))


def camp_add_rmsnorm_plan(x, r, w, h, y, rows: int, cols: int, dtype) -> Plan:
    p = Plan()
    _check("camp_add_rmsnorm_plan", load().camp_add_rmsnorm_plan(
        _ptr(x), _ptr(r), _ptr(w), _ptr(h), _ptr(y), int(rows), int(cols), _dtype(dtype),
        ctypes.byref(p)))
    return p


def camp_add_rmsnorm_with_plan(x, r, w, h, y, rows: int, cols: int, eps: float, dtype,
                               plan: Plan, stream=None) -> None:
    _check("camp_add_rmsnorm_with_plan", load().camp_add_rmsnorm_with_plan(
        _ptr(x), _ptr(r), _ptr(w), _ptr(h), _ptr(y), int(rows), int(cols), float(eps),
        _dtype(dtype), ctypes.byref(plan), _stream(stream)))


def camp_kv_rmsnorm_rope_cache(kv, gamma, sin, cos, slots, cache_n, cache_r, B: int, S: int,
                               Dn: int, Dr: int, num_slots: int, eps: float, dtype,
                               stream=None) -> None:
    _check("camp_kv_rmsnorm_rope_cache", load().camp_kv_rmsnorm_rope_cache(
        _ptr(kv), _ptr(gamma), _ptr(sin), _ptr(cos), _ptr(slots), _ptr(cache_n), _ptr(cache_r),
        int(B), int(S), int(Dn), int(Dr), int(num_slots), float(eps), _dtype(dtype),
        _stream(stream)))


def camp_kv_rmsnorm_rope_cache_plan(kv, gamma, sin, cos, slots, cache_n, cache_r, B: int,
                                    S: int, Dn: int, Dr: int, num_slots: int, dtype) -> Plan:
    p = Plan()
    _check("camp_kv_rmsnorm_rope_cache_plan", load().camp_kv_rmsnorm_rope_cache_plan(
        _ptr(kv), _ptr(gamma), _ptr(sin), _ptr(cos), _ptr(slots), _ptr(cache_n), _ptr(cache_r),
        int(B), int(S), int(Dn), int(Dr), int(num_slots), _dtype(dtype), ctypes.byref(p)))
    return p


def camp_kv_rmsnorm_rope_cache_with_plan(kv, gamma, sin, cos, slots, cache_n, cache_r, B: int,
                                         S: int, Dn: int, Dr: int, num_slots: int, eps: float,
                                         dtype, plan: Plan, stream=None) -> None:
    _check("camp_kv_rmsnorm_rope_cache_with_plan", load().camp_kv_rmsnorm_rope_cache_with_plan(
        _ptr(kv), _ptr(gamma), _ptr(sin), _ptr(cos), _ptr(slots), _ptr(cache_n), _ptr(cache_r),
        int(B), int(S), int(Dn), int(Dr), int(num_slots), float(eps), _dtype(dtype),
        ctypes.byref(plan), _stream(stream)))


def camp_layernorm(x, gamma, beta, y, rows: int, cols: int, eps: float, dtype, stream=None) -> None:
    _check("camp_layernorm", load().camp_layernorm(
        _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), int(rows), int(cols), float(eps),
        _dtype(dtype), _stream(stream)))


def camp_layernorm_wait_probe(x, gamma, beta, y, rows: int, cols: int, eps: float, dtype,
                              wait_ns: int, plan: Plan | None = None, stream=None) -> None:
    """The staged LayerNorm (or the staged or spread kernel of `plan`) with every wait
    bounded by `wait_ns` and each CTA's first row copy left unissued (a diagnostic of the
    bounded waits; see include/camp.h)."""
    _check("camp_layernorm_wait_probe", load().camp_layernorm_wait_probe(
        _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), int(rows), int(cols), float(eps),
        _dtype(dtype), None if plan is None else ctypes.byref(plan), int(wait_ns),
        _stream(stream)))


def camp_rmsnorm_wait_probe(x, w, y, rows: int, cols: int, eps: float, dtype, wait_ns: int,
                            plan: Plan | None = None, stream=None) -> None:
    """The staged RMSNorm (or the staged or spread kernel of `plan`) with every wait bounded
    by `wait_ns` and each CTA's first row copy left unissued (a diagnostic of the bounded
    waits; see include/camp.h)."""
    _check("camp_rmsnorm_wait_probe", load().camp_rmsnorm_wait_probe(
        _ptr(x), _ptr(w), _ptr(y), int(rows), int(cols), float(eps), _dtype(dtype),
        None if plan is None else ctypes.byref(plan), int(wait_ns), _stream(stream)))


def camp_layernorm_plan(x, gamma, beta, y, rows: int, cols: int, dtype) -> Plan:
    p = Plan()
    _check("camp_layernorm_plan", load().camp_layernorm_plan(
        _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), int(rows), int(cols), _dtype(dtype),
        ctypes.byref(p)))
    return p


def camp_layernorm_with_plan(x, gamma, beta, y, rows: int, cols: int, eps: float, dtype,
                             plan: Plan, stream=None) -> None:
    _check("camp_layernorm_with_plan", load().camp_layernorm_with_plan(
        _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), int(rows), int(cols), float(eps),
        _dtype(dtype), ctypes.byref(plan), _stream(stream)))


def camp_rope_interleaved(x, sin, cos, positions, y, tokens: int, H: int, D: int, max_pos: int,
                          dtype, stream=None) -> None:
    _check("camp_rope_interleaved", load().camp_rope_interleaved(
        _ptr(x), _ptr(sin), _ptr(cos), _ptr(positions), _ptr(y), int(tokens), int(H), int(D),
        int(max_pos), _dtype(dtype), _stream(stream)))


def camp_rope_interleaved_plan(x, sin, cos, positions, y, tokens: int, H: int, D: int,
                               max_pos: int, dtype) -> Plan:
    p = Plan()
    _check("camp_rope_interleaved_plan", load().camp_rope_interleaved_plan(
        _ptr(x), _ptr(sin), _ptr(cos), _ptr(positions), _ptr(y), int(tokens), int(H), int(D),
        int(max_pos), _dtype(dtype), ctypes.byref(p)))
    return p


def camp_rope_interleaved_with_plan(x, sin, cos, positions, y, tokens: int, H: int, D: int,
                                    max_pos: int, dtype, plan: Plan, stream=None) -> None:
    _check("camp_rope_interleaved_with_plan", load().camp_rope_interleaved_with_plan(
        _ptr(x), _ptr(sin), _ptr(cos), _ptr(positions), _ptr(y), int(tokens), int(H), int(D),
        int(max_pos), _dtype(dtype), ctypes.byref(plan), _stream(stream)))


def camp_kv_cat_repeat(past, fresh, sin, cos, out, B: int, P: int, S: int, Hk: int, D: int,
                       n_rep: int, dtype, stream=None) -> None:
    _check("camp_kv_cat_repeat", load().camp_kv_cat_repeat(
        _ptr(past), _ptr(fresh), _ptr(sin), _ptr(cos), _ptr(out), int(B), int(P), int(S),
        int(Hk), int(D), int(n_rep), _dtype(dtype), _stream(stream)))


def camp_kv_cat_repeat_plan(past, fresh, sin, cos, out, B: int, P: int, S: int, Hk: int, D: int,
                            n_rep: int, dtype) -> Plan:
    p = Plan()
    _check("camp_kv_cat_repeat_plan", load().camp_kv_cat_repeat_plan(
        _ptr(past), _ptr(fresh), _ptr(sin), _ptr(cos), _ptr(out), int(B), int(P), int(S),
        int(Hk), int(D), int(n_rep), _dtype(dtype), ctypes.byref(p)))
    return p


def camp_kv_cat_repeat_with_plan(past, fresh, sin, cos, out, B: int, P: int, S: int, Hk: int,
                                 D: int, n_rep: int, dtype, plan: Plan, stream=None) -> None:
    _check("camp_kv_cat_repeat_with_plan", load().camp_kv_cat_repeat_with_plan(
        _ptr(past), _ptr(fresh), _ptr(sin), _ptr(cos), _ptr(out), int(B), int(P), int(S),
        int(Hk), int(D), int(n_rep), _dtype(dtype), ctypes.byref(plan), _stream(stream)))


def camp_rope_tables(sin, cos, max_pos: int, D: int, theta: float, stream=None) -> None:
    _check("camp_rope_tables", load().camp_rope_tables(
        _ptr(sin), _ptr(cos), int(max_pos), int(D), float(theta), _stream(stream)))


def camp_rope_qk(q, k, sin, cos, yq, yk, B: int, S: int, Hq: int, Hk: int, D: int, dtype,
                 stream=None) -> None:
    _check("camp_rope_qk", load().camp_rope_qk(
        _ptr(q), _ptr(k), _ptr(sin), _ptr(cos), _ptr(yq), _ptr(yk), int(B), int(S), int(Hq),
        int(Hk), int(D), _dtype(dtype), _stream(stream)))


def camp_rope_qk_plan(q, k, sin, cos, yq, yk, B: int, S: int, Hq: int, Hk: int, D: int,
                      dtype) -> Plan:
    p = Plan()
    _check("camp_rope_qk_plan", load().camp_rope_qk_plan(
        _ptr(q), _ptr(k), _ptr(sin), _ptr(cos), _ptr(yq), _ptr(yk), int(B), int(S), int(Hq),
        int(Hk), int(D), _dtype(dtype), ctypes.byref(p)))
    return p


def camp_rope_qk_with_plan(q, k, sin, cos, yq, yk, B: int, S: int, Hq: int, Hk: int, D: int,
                           dtype, plan: Plan, stream=None) -> None:
    _check("camp_rope_qk_with_plan", load().camp_rope_qk_with_plan(
        _ptr(q), _ptr(k), _ptr(sin), _ptr(cos), _ptr(yq), _ptr(yk), int(B), int(S), int(Hq),
        int(Hk), int(D), _dtype(dtype), ctypes.byref(plan), _stream(stream)))


# ------------------------------------------------------------------ tensor conveniences

def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def rmsnorm(x, w, eps: float = 1e-5, out=None, stream=None):
    """RMSNorm over the last dimension of a contiguous CUDA tensor (bf16, fp16 or fp32)."""
    import torch
    _require(x.is_cuda and x.is_contiguous(), "x must be a contiguous CUDA tensor")
    _require(w.dtype == x.dtype and w.is_contiguous() and w.numel() == x.shape[-1],
             "w must be a contiguous [cols] tensor of x's dtype")
    if out is None:
        out = torch.empty_like(x)
    _require(out.shape == x.shape and out.dtype == x.dtype and out.is_contiguous(),
             "out must match x")
    cols = x.shape[-1] if x.dim() > 0 else 1
    rows = x.numel() // cols if cols else 0
    camp_rmsnorm(x, w, out, rows, cols, eps, x.dtype, stream)
    return out


def rope(x, sin, cos, out=None, stream=None):
    """Rotate-half RoPE of a contiguous CUDA tensor x[B, S, H, D] with fp32 tables [S, D/2]."""
    import torch
    _require(x.is_cuda and x.is_contiguous() and x.dim() == 4, "x must be contiguous [B,S,H,D]")
    B, S, H, D = x.shape
    for t, name in ((sin, "sin"), (cos, "cos")):
        _require(t.dtype == torch.float32 and t.is_contiguous() and tuple(t.shape) == (S, D // 2),
                 f"{name} must be a contiguous fp32 [S, D/2] tensor")
    if out is None:
        out = torch.empty_like(x)
    _require(out.shape == x.shape and out.dtype == x.dtype and out.is_contiguous(),
             "out must match x")
    camp_rope(x, sin, cos, out, B, S, H, D, x.dtype, stream)
    return out


def rope_qk(q, k, sin, cos, out_q=None, out_k=None, stream=None):
    """Rotate-half RoPE of Q[B, S, Hq, D] and K[B, S, Hk, D] with shared fp32 tables, one launch."""
    import torch
    _require(q.is_cuda and k.is_cuda and q.is_contiguous() and k.is_contiguous()
             and q.dim() == 4 and k.dim() == 4, "q and k must be contiguous [B,S,H,D]")
    B, S, Hq, D = q.shape
    _require(k.shape[0] == B and k.shape[1] == S and k.shape[3] == D and k.dtype == q.dtype,
             "k must match q in B, S, D and dtype")
    Hk = k.shape[2]
    for t, name in ((sin, "sin"), (cos, "cos")):
        _require(t.dtype == torch.float32 and t.is_contiguous() and tuple(t.shape) == (S, D // 2),
                 f"{name} must be a contiguous fp32 [S, D/2] tensor")
    out_q = torch.empty_like(q) if out_q is None else out_q
    out_k = torch.empty_like(k) if out_k is None else out_k
    camp_rope_qk(q, k, sin, cos, out_q, out_k, B, S, Hq, Hk, D, q.dtype, stream)
    return out_q, out_k


def add_rmsnorm(x, r, w, eps: float = 1e-5, out_h=None, out_y=None, stream=None):
    """h = x + r and y = RMSNorm(h) * w over the last dimension, in one launch."""
    import torch
    _require(x.is_cuda and x.is_contiguous() and r.shape == x.shape and r.dtype == x.dtype
             and r.is_contiguous(), "x and r must be contiguous CUDA tensors of one shape")
    _require(w.dtype == x.dtype and w.is_contiguous() and w.numel() == x.shape[-1],
             "w must be a contiguous [cols] tensor of x's dtype")
    out_h = torch.empty_like(x) if out_h is None else out_h
    out_y = torch.empty_like(x) if out_y is None else out_y
    cols = x.shape[-1]
    rows = x.numel() // cols
    camp_add_rmsnorm(x, r, w, out_h, out_y, rows, cols, eps, x.dtype, stream)
    return out_h, out_y


def layernorm(x, gamma, beta, eps: float = 1e-5, out=None, stream=None):
    """LayerNorm over the last dimension of a contiguous CUDA tensor (bf16, fp16 or fp32)."""
    import torch
    _require(x.is_cuda and x.is_contiguous(), "x must be a contiguous CUDA tensor")
    for t, name in ((gamma, "gamma"), (beta, "beta")):
        _require(t.dtype == x.dtype and t.is_contiguous() and t.numel() == x.shape[-1],
                 f"{name} must be a contiguous [cols] tensor of x's dtype")
    if out is None:
        out = torch.empty_like(x)
    _require(out.shape == x.shape and out.dtype == x.dtype and out.is_contiguous(),
             "out must match x")
    cols = x.shape[-1] if x.dim() > 0 else 1
    rows = x.numel() // cols if cols else 0
    camp_layernorm(x, gamma, beta, out, rows, cols, eps, x.dtype, stream)
    return out


def kv_cat_repeat(past, fresh, n_rep: int, sin=None, cos=None, out=None, stream=None):
    """out[B, P+S, Hk*n_rep, D] from past[B, P, Hk, D] (or None) and fresh[B, S, Hk, D]:
    concatenated along the sequence, each head repeated n_rep times, the new rows rotated at
    positions P + s when fp32 tables [>= P+S, D/2] are given."""
    import torch
    _require(fresh.is_cuda and fresh.is_contiguous() and fresh.dim() == 4,
             "fresh must be a contiguous CUDA [B, S, Hk, D] tensor")
    B, S, Hk, D = fresh.shape
    P = 0
    if past is not None:
        _require(past.is_contiguous() and past.dim() == 4 and past.dtype == fresh.dtype
                 and past.shape[0] == B and tuple(past.shape[2:]) == (Hk, D),
                 "past must be a contiguous [B, P, Hk, D] tensor of fresh's dtype")
        P = past.shape[1]
    _require((sin is None) == (cos is None), "give both tables or neither")
    for t, name in ((sin, "sin"), (cos, "cos")):
        if t is not None:
            _require(t.dtype == torch.float32 and t.is_contiguous() and t.dim() == 2
                     and t.shape[0] >= P + S and t.shape[1] == D // 2,
                     f"{name} must be a contiguous fp32 [>= P+S, D/2] tensor")
    if out is None:
        out = torch.empty(B, P + S, Hk * n_rep, D, dtype=fresh.dtype, device=fresh.device)
    _require(tuple(out.shape) == (B, P + S, Hk * n_rep, D) and out.dtype == fresh.dtype
             and out.is_contiguous(), "out must be a contiguous [B, P+S, Hk*n_rep, D] tensor")
    camp_kv_cat_repeat(past, fresh, sin, cos, out, B, P, S, Hk, D, n_rep, fresh.dtype, stream)
    return out
