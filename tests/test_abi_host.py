"""Host-side checks of libcamp that need no GPU.

The library must load on a machine without a GPU and export every symbol that
include/camp.h declares. Argument validation and kernel planning run on the host before
any CUDA call, so their results can be checked here with fake (never dereferenced)
pointer values.
"""

from __future__ import annotations

import ctypes
import math
import os
import re

import pytest

from block_memory_bound_gb300 import build, camp

HEADER = os.path.join(build.INCLUDE, "camp.h")

# Fake device addresses: 256-byte aligned and far apart, never dereferenced.
X = 0x7F0000000000
W = 0x7F1000000000
Y = 0x7F2000000000
SIN = 0x7F3000000000
COS = 0x7F4000000000


@pytest.fixture(scope="module")
def lib():
    build.build()
    return camp.load()


def test_exports_every_declared_symbol(lib):
    text = open(HEADER).read()
    declared = set(re.findall(r"CAMP_API\s+[^;(]*?\b(camp_\w+)\s*\(", text))
    assert declared == set(camp.EXPORTS), declared ^ set(camp.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert camp.status_string(camp.SUCCESS) == "success"
    assert camp.status_string(camp.ERR_INVALID_ARG) == "invalid argument"
    assert camp.status_string(camp.ERR_UNSUPPORTED_DTYPE) == "unsupported dtype"
    assert camp.status_string(camp.ERR_RUNTIME) == "CUDA runtime error"
    assert camp.status_string(camp.ERR_NOT_SUPPORTED) == "not supported"
    assert camp.status_string(42) == "unknown status"
    assert camp.camp_last_cuda_error() == 0


def _rms(lib, x=X, w=W, y=Y, rows=4, cols=8, eps=1e-5, dtype=camp.BF16):
    return lib.camp_rmsnorm(x, w, y, rows, cols, ctypes.c_float(eps), dtype, None)


def _rope(lib, x=X, s=SIN, c=COS, y=Y, B=1, S=4, H=2, D=8, dtype=camp.BF16):
    return lib.camp_rope(x, s, c, y, B, S, H, D, dtype, None)


@pytest.mark.parametrize("kw,status", [
    ({"dtype": -1}, camp.ERR_UNSUPPORTED_DTYPE),
    ({"dtype": 2}, camp.ERR_UNSUPPORTED_DTYPE),
    ({"rows": -1}, camp.ERR_INVALID_ARG),
    ({"cols": 0}, camp.ERR_INVALID_ARG),
    ({"cols": -5}, camp.ERR_INVALID_ARG),
    ({"eps": -1e-5}, camp.ERR_INVALID_ARG),
    ({"eps": math.nan}, camp.ERR_INVALID_ARG),
    ({"eps": math.inf}, camp.ERR_INVALID_ARG),
    ({"x": None}, camp.ERR_INVALID_ARG),
    ({"w": None}, camp.ERR_INVALID_ARG),
    ({"y": None}, camp.ERR_INVALID_ARG),
    ({"x": X + 1}, camp.ERR_INVALID_ARG),                       # not element aligned
    ({"y": Y + 2, "dtype": camp.F32}, camp.ERR_INVALID_ARG),
    ({"y": X + 2}, camp.ERR_INVALID_ARG),                       # partial overlap with x
    ({"y": X - 2}, camp.ERR_INVALID_ARG),
    ({"y": W}, camp.ERR_INVALID_ARG),                           # output over the weight
    ({"y": W - 16}, camp.ERR_INVALID_ARG),
    ({"rows": 2**62, "cols": 2**10}, camp.ERR_INVALID_ARG),     # byte count overflows
])
def test_rmsnorm_argument_errors(lib, kw, status):
    assert _rms(lib, **kw) == status


def test_rmsnorm_empty_is_success_without_cuda(lib):
    assert _rms(lib, rows=0) == camp.SUCCESS
    assert _rms(lib, x=None, w=None, y=None, rows=0) == camp.SUCCESS
    # an invalid eps is still reported for an empty call
    assert _rms(lib, rows=0, eps=-1.0) == camp.ERR_INVALID_ARG


@pytest.mark.parametrize("kw,status", [
    ({"dtype": 7}, camp.ERR_UNSUPPORTED_DTYPE),
    ({"D": 7}, camp.ERR_INVALID_ARG),
    ({"D": 0}, camp.ERR_INVALID_ARG),
    ({"D": -2}, camp.ERR_INVALID_ARG),
    ({"B": -1}, camp.ERR_INVALID_ARG),
    ({"S": -1}, camp.ERR_INVALID_ARG),
    ({"H": -3}, camp.ERR_INVALID_ARG),
    ({"x": None}, camp.ERR_INVALID_ARG),
    ({"s": None}, camp.ERR_INVALID_ARG),
    ({"c": None}, camp.ERR_INVALID_ARG),
    ({"y": None}, camp.ERR_INVALID_ARG),
    ({"x": X + 1}, camp.ERR_INVALID_ARG),
    ({"s": SIN + 2}, camp.ERR_INVALID_ARG),                     # tables are fp32
    ({"y": X + 2}, camp.ERR_INVALID_ARG),                       # partial overlap with x
    ({"y": SIN}, camp.ERR_INVALID_ARG),                         # output over a table
    ({"y": COS - 8}, camp.ERR_INVALID_ARG),
    ({"B": 2**40, "S": 2**20, "H": 2**10}, camp.ERR_INVALID_ARG),
])
def test_rope_argument_errors(lib, kw, status):
    assert _rope(lib, **kw) == status


def test_rope_empty_is_success_without_cuda(lib):
    for kw in ({"B": 0}, {"S": 0}, {"H": 0}):
        assert _rope(lib, x=None, s=None, c=None, y=None, **kw) == camp.SUCCESS
    assert _rope(lib, B=0, D=3) == camp.ERR_INVALID_ARG


# ------------------------------------------------------------------ planning

@pytest.mark.parametrize("rows,cols,dtype,expect", [
    # (kernel, vec_bytes, group, per_thread, block, grid)
    # 256 vectors a row: 128 x 2 and 64 x 4 both fit exactly. At 4096 rows 64 x 4 runs in one
    # wave (1024 CTAs <= 152 SMs x 8) and 128 x 2 does not (2048 CTAs); with two waves
    # either way, or one either way, fewer accesses per thread wins
    (4096, 2048, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 64, 4, 256, 1024)),
    (8192, 2048, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 128, 2, 256, 4096)),
    (2048, 2048, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 128, 2, 256, 1024)),
    (16384, 8192, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 256, 4, 256, 16384)),
    # 375 vectors a row: 128 x 3 leaves 9 slots idle, 256 x 2 leaves 137
    (4096, 3000, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 128, 3, 256, 2048)),
    # 64 rows: one row per CTA reaches the most SMs; with no more rows than SMs the launch
    # is latency-bound: the fewest accesses per thread in a group of at most 512 threads
    (64, 2048, "f32", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 1, 512, 64)),
    (1, 8192, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 2, 512, 1)),
    (8, 3000, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 1, 512, 8)),
    (152, 2048, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 256, 1, 256, 152)),
    # past the SMs, up to 2048 rows: 2..4 accesses in groups of up to 512 threads
    (153, 8192, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 2, 512, 153)),
    (2048, 8192, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 2, 512, 2048)),
    (4096, 8192, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 256, 4, 256, 4096)),
    (1, 8, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 32, 1, 256, 1)),
    (64, 3001, "bf16", (camp.KERNEL_RMSNORM_ROWS, 2, 256, 16, 256, 64)),
    # wider rows: one CTA of up to 1024 threads while it holds the row (8192 vectors);
    # past 1024 vectors at most 4 accesses in groups of at most 512 threads...
    (4096, 12288, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 3, 512, 4096)),
    (4096, 16384, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 4, 512, 4096)),
    (2048, 24576, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 6, 512, 2048)),
    (1024, 32768, "bf16", (camp.KERNEL_RMSNORM_ROWS, 16, 512, 8, 512, 1024)),
    # ...then (past 4096 vectors) rows staged in shared memory by persistent clusters:
    # group = vectors a CTA (about 1024), per_thread = buffers (3; 2 with 16 CTAs),
    # grid = the clusters that fit (estimated), at most one per row, x the cluster size
    (5, 65536, "bf16", (camp.KERNEL_RMSNORM_STAGED, 16, 1024, 3, 256, 40, 8)),
    (5, 65544, "bf16", (camp.KERNEL_RMSNORM_STAGED, 16, 513, 2, 256, 80, 16)),
    (256, 131072, "bf16", (camp.KERNEL_RMSNORM_STAGED, 16, 1024, 2, 256, 608, 16)),
    (2, 262144, "bf16", (camp.KERNEL_RMSNORM_STAGED, 16, 2048, 2, 256, 32, 16)),
    (7, 32768, "f32", (camp.KERNEL_RMSNORM_STAGED, 16, 1024, 3, 256, 56, 8)),
    # past 16 x 2048 vectors: a cluster of CTAs of 512 threads per row, each CTA's chunk
    # held in shared memory, one buffer, the smallest cluster whose chunks hold at most 4700
    # vectors (else 16), doubled while the rows' CTAs number under 76; grid = the clusters
    # that fit (3 CTAs an SM at most), at most one per row, x the cluster
    (3, 131080, "f32", (camp.KERNEL_RMSNORM_SPREAD, 16, 2049, 1, 512, 48, 16)),   # 8 x 3 < 76
    (2, 262152, "bf16", (camp.KERNEL_RMSNORM_SPREAD, 16, 2049, 1, 512, 32, 16)),
    (512, 300000, "bf16", (camp.KERNEL_RMSNORM_SPREAD, 16, 4688, 1, 512, 456, 8)),
    (64, 524296, "bf16", (camp.KERNEL_RMSNORM_SPREAD, 16, 4097, 1, 512, 448, 16)),
    (40, 1600000, "bf16", (camp.KERNEL_RMSNORM_SPREAD, 16, 12500, 1, 512, 144, 16)),
    # past what a cluster's shared memory holds, or element accesses: two sweeps in one CTA
    (3, 2000000, "bf16", (camp.KERNEL_RMSNORM_WIDE, 16, 1024, 0, 1024, 3, 1)),
    (5, 16385, "f32", (camp.KERNEL_RMSNORM_WIDE, 4, 1024, 0, 1024, 5, 1)),
])
def test_rmsnorm_plans(lib, rows, cols, dtype, expect):
    p = camp.camp_rmsnorm_plan(X, W, Y, rows, cols, dtype)
    got = (p.kernel, p.vec_bytes, p.group, p.per_thread, p.block, p.grid, p.cluster)
    assert got == (expect if len(expect) == 7 else expect + (1,))


def test_rmsnorm_plan_misaligned_pointer_uses_element_accesses(lib):
    p = camp.camp_rmsnorm_plan(X + 2, W, Y + 2, 4, 2048, "bf16")
    assert p.vec_bytes == 2
    p = camp.camp_rmsnorm_plan(X, W + 4, Y, 4, 2048, "f32")
    assert p.vec_bytes == 4


@pytest.mark.parametrize("B,S,H,D,dtype,expect", [
    # (kernel, vec_bytes, heads per thread, grid)
    # Q: 2 heads per thread, 16 x 4 threads per position, 4 positions per CTA
    (1, 4096, 32, 64, "bf16", (camp.KERNEL_ROPE, 16, 2, 1024)),
    (1, 4096, 8, 64, "bf16", (camp.KERNEL_ROPE, 16, 2, 256)),
    # many positions: 4 heads per thread
    (1, 65536, 32, 128, "bf16", (camp.KERNEL_ROPE, 16, 4, 16384)),
    (1, 65536, 6, 128, "bf16", (camp.KERNEL_ROPE, 16, 2, 6554)),
    # odd head count: 1 head per thread
    (2, 3, 5, 6, "bf16", (camp.KERNEL_ROPE, 2, 1, 1)),
    # no more positions than SMs: the most threads per position (narrow accesses, 1 head
    # per thread), accesses of at least one pair
    (1, 4, 6, 12, "bf16", (camp.KERNEL_ROPE, 4, 1, 1)),
    (1, 4, 6, 24, "f32", (camp.KERNEL_ROPE, 8, 1, 1)),
    (1, 8, 32, 64, "bf16", (camp.KERNEL_ROPE, 8, 1, 8)),        # 256 threads a position
    (1, 64, 8, 128, "bf16", (camp.KERNEL_ROPE, 4, 1, 64)),
    (1, 152, 32, 128, "bf16", (camp.KERNEL_ROPE, 16, 1, 152)),
    # past the SMs, while the bandwidth choice would leave fewer than 128 CTAs: the variant
    # with the smallest grid of at least 128 CTAs
    (1, 153, 32, 128, "bf16", (camp.KERNEL_ROPE, 16, 1, 153)),
    (1, 256, 8, 64, "bf16", (camp.KERNEL_ROPE, 4, 1, 128)),
    (1, 512, 8, 64, "bf16", (camp.KERNEL_ROPE, 8, 1, 128)),
    (1, 1024, 8, 64, "bf16", (camp.KERNEL_ROPE, 16, 1, 128)),
    (1, 512, 32, 64, "bf16", (camp.KERNEL_ROPE, 16, 2, 128)),     # already 128 CTAs
    # a position needs more than one CTA: the flat kernel
    (1, 4, 1024, 256, "bf16", (camp.KERNEL_ROPE_FLAT, 16, 2, 128)),
])
def test_rope_plans(lib, B, S, H, D, dtype, expect):
    p = camp.camp_rope_plan(X, SIN, COS, Y, B, S, H, D, dtype)
    assert p.block == 256 and p.cluster == 1
    assert (p.kernel, p.vec_bytes, p.group, p.grid) == expect


def test_with_plan_rejects_plans_that_do_not_fit(lib):
    bad = [
        camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=16, group=32, per_thread=1),  # too small
        camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=16, group=48, per_thread=8),  # not compiled
        camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=8, group=32, per_thread=8),   # not compiled
        camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=3, group=32, per_thread=8),
        camp.Plan(kernel=camp.KERNEL_ROPE, vec_bytes=16, group=4, per_thread=0),
        camp.Plan(kernel=99, vec_bytes=16, group=32, per_thread=8),
    ]
    for p in bad:
        st = lib.camp_rmsnorm_with_plan(X, W, Y, 4, 2048, ctypes.c_float(1e-5), camp.BF16,
                                        ctypes.byref(p), None)
        assert st == camp.ERR_NOT_SUPPORTED, p
    # 16-byte accesses are refused when a pointer is only element aligned
    p = camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=16, group=64, per_thread=4)
    st = lib.camp_rmsnorm_with_plan(X + 2, W, Y, 4, 2048, ctypes.c_float(1e-5), camp.BF16,
                                    ctypes.byref(p), None)
    assert st == camp.ERR_NOT_SUPPORTED
    rp = camp.Plan(kernel=camp.KERNEL_ROPE, vec_bytes=16, group=3)
    st = lib.camp_rope_with_plan(X, SIN, COS, Y, 1, 4, 6, 64, camp.BF16, ctypes.byref(rp), None)
    assert st == camp.ERR_NOT_SUPPORTED
    rp = camp.Plan(kernel=camp.KERNEL_ROPE, vec_bytes=16, group=2)
    st = lib.camp_rope_with_plan(X, SIN, COS, Y, 1, 4, 6, 6, camp.BF16, ctypes.byref(rp), None)
    assert st == camp.ERR_NOT_SUPPORTED        # a 3-element half is not 16-byte vectors


def test_binding_raises_on_errors(lib):
    with pytest.raises(camp.CampError) as e:
        camp.camp_rmsnorm(X, W, Y, 4, 0, 1e-5, "bf16", 0)
    assert e.value.status == camp.ERR_INVALID_ARG
    with pytest.raises(camp.CampError) as e:
        camp.camp_rope(X, SIN, COS, Y, 1, 4, 2, 7, "bf16", 0)
    assert e.value.status == camp.ERR_INVALID_ARG


def test_fast_division_algorithm():
    # The RoPE kernel derives the table row with Granlund-Montgomery division by an
    # invariant: l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
    # n / d = (umulhi(m, n) + n) >> l. Check the algorithm on edge and random cases.
    import random
    rng = random.Random(5)
    divisors = [1, 2, 3, 5, 7, 31, 32, 33, 4095, 4096, 4097, 65536, 70001, 2**31 - 1, 2**31,
                2**31 + 1, 2**32 - 1] + [rng.randrange(1, 2**32) for _ in range(200)]
    for d in divisors:
        l = 0
        while (1 << l) < d:
            l += 1
        m = ((1 << 32) * ((1 << l) - d)) // d + 1
        assert 0 < m < (1 << 32)
        ns = [0, 1, d - 1, d, d + 1, 2**32 - 1, 2**32 - 2] + [rng.randrange(2**32) for _ in range(300)]
        for n in ns:
            if n >= 2**32:
                continue
            t = (m * n) >> 32
            assert (t + n) >> l == n // d, (n, d)


# ------------------------------------------------------------------ fused Q + K RoPE

K_ = 0x7F5000000000
YQ = 0x7F6000000000
YK = 0x7F7000000000


def _qk(lib, q=X, k=K_, s=SIN, c=COS, yq=YQ, yk=YK, B=1, S=4, Hq=4, Hk=2, D=8,
        dtype=camp.BF16):
    return lib.camp_rope_qk(q, k, s, c, yq, yk, B, S, Hq, Hk, D, dtype, None)


@pytest.mark.parametrize("kw,status", [
    ({"dtype": 5}, camp.ERR_UNSUPPORTED_DTYPE),
    ({"D": 5}, camp.ERR_INVALID_ARG),
    ({"Hq": -1}, camp.ERR_INVALID_ARG),
    ({"Hk": -1}, camp.ERR_INVALID_ARG),
    ({"q": None}, camp.ERR_INVALID_ARG),
    ({"k": None}, camp.ERR_INVALID_ARG),
    ({"yq": None}, camp.ERR_INVALID_ARG),
    ({"yk": None}, camp.ERR_INVALID_ARG),
    ({"s": None}, camp.ERR_INVALID_ARG),
    ({"k": K_ + 1}, camp.ERR_INVALID_ARG),                 # misaligned
    ({"yq": K_}, camp.ERR_INVALID_ARG),                    # Q's output over K's input
    ({"yk": X + 16}, camp.ERR_INVALID_ARG),                # K's output inside Q's input
    ({"yk": YQ + 32}, camp.ERR_INVALID_ARG),               # the two outputs overlap
    ({"yk": COS}, camp.ERR_INVALID_ARG),                   # an output over a table
    ({"yq": X + 2}, camp.ERR_INVALID_ARG),                 # partial in-place overlap
])
def test_rope_qk_argument_errors(lib, kw, status):
    assert _qk(lib, **kw) == status


def test_rope_qk_empty_and_single_tensor_calls_need_no_cuda(lib):
    assert _qk(lib, q=None, k=None, s=None, c=None, yq=None, yk=None, B=0) == camp.SUCCESS
    assert _qk(lib, q=None, k=None, s=None, c=None, yq=None, yk=None, Hq=0, Hk=0) == camp.SUCCESS
    # with no heads, a tensor's pointers are not inspected (this one would overlap)
    p = camp.camp_rope_qk_plan(X, X + 2, SIN, COS, YQ, X + 2, 1, 4096, 32, 0, 64, "bf16")
    assert (p.kernel, p.group, p.grid) == (camp.KERNEL_ROPE, 2, 1024)
    p = camp.camp_rope_qk_plan(X + 2, K_, SIN, COS, X + 2, YK, 1, 4096, 0, 8, 64, "bf16")
    assert (p.kernel, p.vec_bytes, p.group, p.grid) == (camp.KERNEL_ROPE, 16, 2, 256)


@pytest.mark.parametrize("B,S,Hq,Hk,D,expect", [
    # Q 32 + K 8 heads of 64, 2 heads per thread: (16 + 4) x 4 = 80 threads a position,
    # 3 positions per CTA
    (1, 4096, 32, 8, 64, (camp.KERNEL_ROPE, 16, 2, 1366)),
    (2, 128, 14, 2, 128, (camp.KERNEL_ROPE, 16, 1, 128)),    # 64 CTAs with 2 heads: fill to 128
    (1, 65536, 32, 8, 128, (camp.KERNEL_ROPE, 16, 4, 21846)),
    (1, 16, 3, 1, 64, (camp.KERNEL_ROPE, 4, 1, 4)),         # decode size: 64 threads a position
    (1, 8, 32, 8, 64, (camp.KERNEL_ROPE, 16, 1, 8)),         # 160 threads: the widest of 3 ties
    # the heads of a position do not fit one CTA: two launches (K alone takes the decode rule)
    (1, 4, 1024, 8, 256, (camp.KERNEL_ROPE_SPLIT, 16, 2, 132)),
])
def test_rope_qk_plans(lib, B, S, Hq, Hk, D, expect):
    p = camp.camp_rope_qk_plan(X, K_, SIN, COS, YQ, YK, B, S, Hq, Hk, D, "bf16")
    assert (p.kernel, p.vec_bytes, p.group, p.grid) == expect


def test_rope_qk_with_plan_accepts_only_the_fused_launch(lib):
    for p in (camp.Plan(kernel=camp.KERNEL_ROPE_FLAT, vec_bytes=16, group=2),
              camp.Plan(kernel=camp.KERNEL_ROPE_SPLIT, vec_bytes=16, group=2),
              camp.Plan(kernel=camp.KERNEL_ROPE, vec_bytes=16, group=3)):
        st = lib.camp_rope_qk_with_plan(X, K_, SIN, COS, YQ, YK, 1, 4, 4, 2, 64, camp.BF16,
                                        ctypes.byref(p), None)
        assert st == camp.ERR_NOT_SUPPORTED


def test_cluster_plans_that_do_not_fit_are_refused(lib):
    for cl, nv, cols in ((3, 4, 8192), (2, 5, 8192), (2, 1, 8192), (32, 1, 8192)):
        p = camp.Plan(kernel=camp.KERNEL_RMSNORM_CLUSTER, vec_bytes=16, per_thread=nv, cluster=cl)
        st = lib.camp_rmsnorm_with_plan(X, W, Y, 4, cols, ctypes.c_float(1e-5), camp.BF16,
                                        ctypes.byref(p), None)
        assert st == camp.ERR_NOT_SUPPORTED, (cl, nv)
    # the cluster kernel uses 16-byte accesses only
    p = camp.Plan(kernel=camp.KERNEL_RMSNORM_CLUSTER, vec_bytes=2, per_thread=4, cluster=2)
    st = lib.camp_rmsnorm_with_plan(X, W, Y, 4, 2048, ctypes.c_float(1e-5), camp.BF16,
                                    ctypes.byref(p), None)
    assert st == camp.ERR_NOT_SUPPORTED


# ------------------------------------------------------------------ fused residual add + RMSNorm

R_ = 0x7F8000000000
H_ = 0x7F9000000000


def _addrms(lib, x=X, r=R_, w=W, h=H_, y=Y, rows=4, cols=8, eps=1e-5, dtype=camp.BF16):
    return lib.camp_add_rmsnorm(x, r, w, h, y, rows, cols, ctypes.c_float(eps), dtype, None)


@pytest.mark.parametrize("kw,status", [
    ({"dtype": 9}, camp.ERR_UNSUPPORTED_DTYPE),
    ({"cols": 0}, camp.ERR_INVALID_ARG),
    ({"eps": -1.0}, camp.ERR_INVALID_ARG),
    ({"r": None}, camp.ERR_INVALID_ARG),
    ({"h": None}, camp.ERR_INVALID_ARG),
    ({"r": R_ + 1}, camp.ERR_INVALID_ARG),              # misaligned
    ({"h": Y}, camp.ERR_INVALID_ARG),                   # the two outputs coincide
    ({"h": Y + 8}, camp.ERR_INVALID_ARG),               # ...or overlap
    ({"h": X + 2}, camp.ERR_INVALID_ARG),               # partial overlap with an input
    ({"y": R_ - 4}, camp.ERR_INVALID_ARG),
    ({"h": W}, camp.ERR_INVALID_ARG),                   # output over the weight
])
def test_add_rmsnorm_argument_errors(lib, kw, status):
    assert _addrms(lib, **kw) == status


def test_add_rmsnorm_exact_aliases_are_accepted(lib):
    # h == r (residual updated in place) with y == x, and the other way round; planning
    # needs no CUDA, so a plan proves the arguments were accepted.
    for h, y in ((R_, X), (X, R_), (R_, Y), (H_, X)):
        p = camp.camp_add_rmsnorm_plan(X, R_, W, h, y, 4096, 2048, "bf16")
        assert p.kernel == camp.KERNEL_RMSNORM_ROWS


@pytest.mark.parametrize("rows,cols,expect", [
    # the add path: 2 accesses a thread in groups of up to 512 threads, and past 1024
    # vectors a row 1024-thread groups (2 accesses, else at most 4; fewest at decode sizes)
    (4096, 2048, (camp.KERNEL_RMSNORM_ROWS, 16, 128, 2, 1)),
    (16384, 8192, (camp.KERNEL_RMSNORM_ROWS, 16, 512, 2, 1)),
    (1024, 3000, (camp.KERNEL_RMSNORM_ROWS, 16, 256, 2, 1)),
    (8, 8192, (camp.KERNEL_RMSNORM_ROWS, 16, 512, 2, 1)),
    (512, 12288, (camp.KERNEL_RMSNORM_ROWS, 16, 1024, 2, 1)),
    (4096, 16384, (camp.KERNEL_RMSNORM_ROWS, 16, 1024, 2, 1)),
    (1, 16384, (camp.KERNEL_RMSNORM_ROWS, 16, 1024, 2, 1)),
    (2048, 24576, (camp.KERNEL_RMSNORM_ROWS, 16, 1024, 3, 1)),
    (152, 32768, (camp.KERNEL_RMSNORM_ROWS, 16, 1024, 4, 1)),
    (8192, 32768, (camp.KERNEL_RMSNORM_ROWS, 16, 1024, 4, 1)),
    # past 4096 vectors a row the add path stages x and r in shared memory: 4 CTAs of 3
    # buffers up to 6144 vectors, and up to 8192 with fewer than 1024 rows; 16 CTAs of 3
    # buffers at 6144..8192 vectors from 1024 rows on; past 8192 the plain rule
    (64, 40000, (camp.KERNEL_RMSNORM_STAGED, 16, 1250, 3, 4)),
    (4096, 40000, (camp.KERNEL_RMSNORM_STAGED, 16, 1250, 3, 4)),
    (512, 65536, (camp.KERNEL_RMSNORM_STAGED, 16, 2048, 3, 4)),
    (1024, 65536, (camp.KERNEL_RMSNORM_STAGED, 16, 512, 3, 16)),
    (1024, 50000, (camp.KERNEL_RMSNORM_STAGED, 16, 391, 3, 16)),
    (512, 131072, (camp.KERNEL_RMSNORM_STAGED, 16, 1024, 2, 16)),
])
def test_add_rmsnorm_plans(lib, rows, cols, expect):
    p = camp.camp_add_rmsnorm_plan(X, R_, W, H_, Y, rows, cols, "bf16")
    assert (p.kernel, p.vec_bytes, p.group, p.per_thread, p.cluster) == expect


def test_add_rmsnorm_unbuilt_variant_is_refused(lib):
    p = camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=16, group=1024, per_thread=8)
    st = lib.camp_add_rmsnorm_with_plan(X, R_, W, H_, Y, 4, 65536, ctypes.c_float(1e-5),
                                        camp.BF16, ctypes.byref(p), None)
    assert st == camp.ERR_NOT_SUPPORTED


# ------------------------------------------------------------------ KV RMSNorm + RoPE + cache

KVP = [0x7E0000000000 + i * 0x1000000000 for i in range(7)]   # kv, gamma, sin, cos, slots, cn, cr


def _kv(lib, ptrs=None, B=1, S=16, Dn=512, Dr=64, ns=64, eps=1e-5, dtype=camp.BF16):
    p = list(KVP if ptrs is None else ptrs)
    return lib.camp_kv_rmsnorm_rope_cache(*p, B, S, Dn, Dr, ns, ctypes.c_float(eps), dtype, None)


@pytest.mark.parametrize("change,kw,status", [
    ({}, {"dtype": 4}, camp.ERR_UNSUPPORTED_DTYPE),
    ({}, {"Dr": 63}, camp.ERR_INVALID_ARG),
    ({}, {"Dr": 0}, camp.ERR_INVALID_ARG),
    ({}, {"Dn": 0}, camp.ERR_INVALID_ARG),
    ({}, {"ns": -1}, camp.ERR_INVALID_ARG),
    ({}, {"eps": math.nan}, camp.ERR_INVALID_ARG),
    ({4: None}, {}, camp.ERR_INVALID_ARG),                      # no slots
    ({4: KVP[4] + 4}, {}, camp.ERR_INVALID_ARG),                # slots not 8-byte aligned
    ({5: KVP[0]}, {}, camp.ERR_INVALID_ARG),                    # cache over kv
    ({6: KVP[5] + 64}, {}, camp.ERR_INVALID_ARG),               # the caches overlap
    ({6: KVP[2]}, {}, camp.ERR_INVALID_ARG),                    # cache over a table
    ({}, {"Dn": 4096}, camp.ERR_NOT_SUPPORTED),                 # norm part wider than a warp holds
])
def test_kv_cache_argument_errors(lib, change, kw, status):
    ptrs = list(KVP)
    for i, v in change.items():
        ptrs[i] = v
    assert _kv(lib, ptrs, **kw) == status


@pytest.mark.parametrize("dtype,Dn,Dr,expect", [
    # (vec_bytes, per_thread, group = rope bytes per half and lane)
    # bf16 Dr 64: 64 bytes a half -> 4-byte accesses (one pair) over 16 lanes
    ("bf16", 512, 64, (16, 2, 4)),
    ("bf16", 512, 128, (16, 2, 4)),      # 32 lanes
    ("bf16", 512, 256, (16, 2, 8)),      # 4 bytes would need 64 lanes
    ("bf16", 2048, 512, (16, 8, 16)),
    ("f32", 512, 64, (16, 4, 8)),        # fp32 pairs: 8 bytes
    ("f32", 1024, 256, (16, 8, 16)),
    ("bf16", 33, 6, (2, 2, 2)),          # odd widths: element accesses for both parts
])
def test_kv_cache_plans(lib, dtype, Dn, Dr, expect):
    p = camp.camp_kv_rmsnorm_rope_cache_plan(*KVP, 1, 65536, Dn, Dr, 131072, dtype)
    assert p.kernel == camp.KERNEL_KV_CACHE
    assert (p.vec_bytes, p.per_thread, p.group) == expect
    assert p.grid == 8192


def test_kv_cache_plan_edges(lib):
    assert _kv(lib, B=0) == camp.SUCCESS
    assert _kv(lib, Dr=1024) == camp.ERR_NOT_SUPPORTED              # 16 bytes x 32 lanes < a half
    # a rope cache that is not 4-byte aligned sends both parts to element accesses
    ptrs = list(KVP)
    ptrs[6] += 2
    p = camp.camp_kv_rmsnorm_rope_cache_plan(*ptrs, 1, 16, 512, 64, 64, "bf16")
    assert (p.vec_bytes, p.per_thread, p.group) == (2, 16, 2)
    # forced plans: a rope width that does not cover a half, or that is not built
    for vb, nvn, rb, dtype in ((16, 2, 4, "bf16"), (16, 4, 4, "f32"), (16, 2, 2, "bf16")):
        plan = camp.Plan(kernel=camp.KERNEL_KV_CACHE, vec_bytes=vb, per_thread=nvn, group=rb)
        Dr = 512 if rb == 4 and dtype == "bf16" else 64
        st = lib.camp_kv_rmsnorm_rope_cache_with_plan(
            *KVP, 1, 16, 512, Dr, 64, ctypes.c_float(1e-5), camp.BF16 if dtype == "bf16" else camp.F32,
            ctypes.byref(plan), None)
        assert st == camp.ERR_NOT_SUPPORTED, (vb, nvn, rb, dtype)


# ------------------------------------------------------------------ interleaved RoPE, tables

ILP = [0x7D0000000000 + i * 0x1000000000 for i in range(5)]   # x, sin, cos, positions, y


@pytest.mark.parametrize("change,kw,status", [
    ({}, {"dtype": 6}, camp.ERR_UNSUPPORTED_DTYPE),
    ({}, {"D": 7}, camp.ERR_INVALID_ARG),
    ({}, {"mp": -1}, camp.ERR_INVALID_ARG),
    ({3: None}, {}, camp.ERR_INVALID_ARG),
    ({3: ILP[3] + 2}, {}, camp.ERR_INVALID_ARG),             # positions are int32
    ({4: ILP[3]}, {}, camp.ERR_INVALID_ARG),                 # output over the positions
    ({4: ILP[0] + 4}, {}, camp.ERR_INVALID_ARG),             # partial in-place overlap
    ({0: ILP[0] + 2, 4: ILP[4] + 2}, {}, camp.ERR_NOT_SUPPORTED),   # not pair-aligned (bf16)
    ({}, {"H": 128, "D": 256}, camp.ERR_NOT_SUPPORTED),      # a token needs more than one CTA
])
def test_rope_interleaved_argument_errors(lib, change, kw, status):
    p = list(ILP)
    for i, v in change.items():
        p[i] = v
    a = {"T": 16, "H": 4, "D": 64, "mp": 32, "dtype": camp.BF16}
    a.update(kw)
    assert lib.camp_rope_interleaved(*p, a["T"], a["H"], a["D"], a["mp"], a["dtype"], None) == status


def test_rope_interleaved_plans(lib):
    # 32 heads of 128: 4 heads a thread, 8 x 16 = 128 threads a token, 2 tokens a CTA
    p = camp.camp_rope_interleaved_plan(*ILP, 65536, 32, 128, 131072, "bf16")
    assert (p.kernel, p.vec_bytes, p.group, p.grid) == (camp.KERNEL_ROPE_INTERLEAVED, 16, 4, 32768)
    p = camp.camp_rope_interleaved_plan(*ILP, 1000, 5, 6, 16, "bf16")     # odd head count
    assert (p.vec_bytes, p.group, p.grid) == (4, 1, 59)   # no variant reaches 128 CTAs
    p = camp.camp_rope_interleaved_plan(*ILP, 4000, 6, 64, 16, "bf16")    # even, not 4k
    assert (p.vec_bytes, p.group, p.grid) == (16, 2, 400)
    # fewer than 128 CTAs: the smallest grid of at least 128 (1000 x 6 x 64: 2 heads a
    # thread would give 100 CTAs)
    p = camp.camp_rope_interleaved_plan(*ILP, 1000, 6, 64, 16, "bf16")
    assert (p.vec_bytes, p.group, p.grid) == (16, 1, 200)
    p = camp.camp_rope_interleaved_plan(*ILP, 1000, 64, 128, 16, "bf16")  # 4 heads: 256 threads
    assert p.group == 4
    p = camp.camp_rope_interleaved_plan(*ILP, 1000, 128, 128, 16, "bf16")  # 4 heads: 512 threads
    assert p.group == 8
    # decode sizes (no more tokens than SMs): the most threads a token within one CTA
    p = camp.camp_rope_interleaved_plan(*ILP, 16, 6, 64, 16, "bf16")      # 6 x 32 = 192
    assert (p.vec_bytes, p.group, p.grid) == (4, 1, 16)
    p = camp.camp_rope_interleaved_plan(*ILP, 16, 32, 128, 16, "bf16")    # 16 x 16 = 256
    assert (p.vec_bytes, p.group, p.grid) == (16, 2, 16)
    p = camp.camp_rope_interleaved_plan(*ILP, 16, 128, 128, 16, "bf16")   # 16 x 16 = 256
    assert (p.vec_bytes, p.group, p.grid) == (16, 8, 16)


def test_rope_tables_argument_errors(lib):
    S_, C_ = ILP[1], ILP[2]
    for args in ((S_, C_, 16, 7, 1e4), (S_, C_, -1, 8, 1e4), (S_, C_, 16, 8, 0.0),
                 (S_, C_, 16, 8, math.inf), (None, C_, 16, 8, 1e4), (S_, S_ + 8, 16, 8, 1e4)):
        assert lib.camp_rope_tables(*args, None) == camp.ERR_INVALID_ARG
    assert lib.camp_rope_tables(None, None, 0, 8, 1e4, None) == camp.SUCCESS


# ------------------------------------------------------------------ LayerNorm

BETA = 0x7FA000000000


def _ln(lib, x=X, g=W, b=BETA, y=Y, rows=4, cols=8, eps=1e-5, dtype=camp.BF16):
    return lib.camp_layernorm(x, g, b, y, rows, cols, ctypes.c_float(eps), dtype, None)


@pytest.mark.parametrize("kw,status", [
    ({"dtype": 4}, camp.ERR_UNSUPPORTED_DTYPE),
    ({"cols": 0}, camp.ERR_INVALID_ARG),
    ({"rows": -2}, camp.ERR_INVALID_ARG),
    ({"eps": -1.0}, camp.ERR_INVALID_ARG),
    ({"eps": math.nan}, camp.ERR_INVALID_ARG),
    ({"g": None}, camp.ERR_INVALID_ARG),
    ({"b": None}, camp.ERR_INVALID_ARG),
    ({"b": BETA + 1}, camp.ERR_INVALID_ARG),            # not element aligned
    ({"y": BETA}, camp.ERR_INVALID_ARG),                # output over beta
    ({"y": BETA - 8}, camp.ERR_INVALID_ARG),
    ({"y": W}, camp.ERR_INVALID_ARG),                   # output over gamma
    ({"y": X + 2}, camp.ERR_INVALID_ARG),               # partial overlap with x
])
def test_layernorm_argument_errors(lib, kw, status):
    assert _ln(lib, **kw) == status


def test_layernorm_empty_and_in_place(lib):
    assert _ln(lib, x=None, g=None, b=None, y=None, rows=0) == camp.SUCCESS
    assert _ln(lib, rows=0, eps=-1.0) == camp.ERR_INVALID_ARG
    p = camp.camp_layernorm_plan(X, W, BETA, X, 4096, 2048, "bf16")   # y == x is accepted
    assert p.kernel == camp.KERNEL_LAYERNORM_ROWS


@pytest.mark.parametrize("rows,cols,dtype", [
    (16384, 8192, "bf16"), (4096, 3000, "bf16"), (64, 2048, "f32"),
    (1, 8, "bf16"), (64, 3001, "bf16"), (3, 8192, "f32"), (4096, 1024, "bf16"),
])
def test_layernorm_plans_follow_the_rmsnorm_rows_chooser(lib, rows, cols, dtype):
    # the same register-resident row mapping as RMSNorm: where neither the one-wave test
    # nor the many-wave rule separates them, the same group and accesses a thread
    p = camp.camp_layernorm_plan(X, W, BETA, Y, rows, cols, dtype)
    q = camp.camp_rmsnorm_plan(X, W, Y, rows, cols, dtype)
    assert q.kernel == camp.KERNEL_RMSNORM_ROWS
    assert p.kernel == camp.KERNEL_LAYERNORM_ROWS
    assert (p.vec_bytes, p.group, p.per_thread, p.block, p.grid, p.cluster) == \
        (q.vec_bytes, q.group, q.per_thread, q.block, q.grid, 1)


def test_layernorm_keeps_the_smaller_group_past_1024_vectors(lib):
    # outside the 2-4 accesses band RMSNorm takes at most 4 accesses in groups of at most
    # 512 threads; LayerNorm (two reductions a row) keeps the smaller group
    for cols, ln, rms in ((12288, (256, 6), (512, 3)), (16384, (256, 8), (512, 4))):
        p = camp.camp_layernorm_plan(X, W, BETA, Y, 4096, cols, "bf16")
        q = camp.camp_rmsnorm_plan(X, W, Y, 4096, cols, "bf16")
        assert (p.kernel, p.group, p.per_thread) == (camp.KERNEL_LAYERNORM_ROWS,) + ln
        assert (q.kernel, q.group, q.per_thread) == (camp.KERNEL_RMSNORM_ROWS,) + rms


@pytest.mark.parametrize("rows,cols,dtype,cluster,chunk,rps", [
    (7, 32768, "f32", 8, 1024, 2),         # two rows a step with chunks of 1024
    (1024, 16384, "f32", 4, 1024, 2),
    (4, 32768, "f32", 8, 1024, 2),
    (256, 65536, "f32", 8, 2048, 1),       # ... but not with a cluster of 16
    (1024, 12288, "f32", 4, 768, 2),       # 0.75 full, but one spread CTA would hold 3072
    (4, 32776, "f32", 8, 1025, 1),         # 0.50 full, but 4 rows split spread chunks to 513
])
def test_fp32_layernorm_stages_rows_past_4096_vectors(lib, rows, cols, dtype, cluster, chunk,
                                                      rps):
    # fp32 rows past 4096 vectors (2048 with at most 1024 rows) are staged in shared memory,
    # 2 buffers (each carries the row's first 16 bytes): two rows a step with chunks of at
    # most 1024 vectors where a cluster of at most 8 gives them, otherwise one row a step
    # with the smallest cluster whose CTA chunks hold at most 2048 vectors
    p = camp.camp_layernorm_plan(X, W, BETA, Y, rows, cols, dtype)
    assert (p.kernel, p.vec_bytes, p.cluster, p.group, p.block, p.per_thread,
            p.rows_per_step) == (camp.KERNEL_LAYERNORM_STAGED, 16, cluster, chunk, 256, 2, rps)


@pytest.mark.parametrize("rows,cols,dtype,cluster,chunk,grid", [
    (64, 262144, "bf16", 8, 4096, 456),    # 3 CTAs an SM: 57 clusters of 8
    (1024, 65536, "f16", 2, 4096, 456),
    (1024, 30720, "bf16", 1, 3840, 456),   # few rows, 3840 vectors
    (1024, 24576, "bf16", 1, 3072, 456),
    (512, 140000, "bf16", 4, 4375, 456),
    (256, 200000, "bf16", 8, 3125, 456),   # 4 CTAs would hold 6250
    (5, 65536, "bf16", 16, 512, 80),       # 5 rows x 2 CTAs: split to 16 a row
    (4, 32768, "bf16", 16, 256, 64),
])
def test_16bit_layernorm_spreads_rows_past_4096_vectors(lib, rows, cols, dtype, cluster,
                                                        chunk, grid):
    # in 16-bit storage the same rows take the spread kernel: one buffer, the smallest
    # cluster whose chunks hold at most 4700 vectors, doubled while the rows' CTAs number
    # under 76; grid = 3 CTAs an SM at most, one cluster a row at most
    p = camp.camp_layernorm_plan(X, W, BETA, Y, rows, cols, dtype)
    assert (p.kernel, p.vec_bytes, p.cluster, p.group, p.block, p.per_thread, p.grid) == \
        (camp.KERNEL_LAYERNORM_SPREAD, 16, cluster, chunk, 512, 1, grid)


@pytest.mark.parametrize("rows,cols,staged_chunk,cluster,chunk,grid", [
    (512, 70000, 1094, 4, 4375, 304),      # 1094 vectors in 8 x 256 slots: 0.53 full
    (1024, 40000, 1250, 2, 5000, 304),     # 0.61 full
    (512, 32776, 1025, 2, 4097, 304),      # 0.50 full
])
def test_fp32_layernorm_ragged_staged_chunks_take_the_spread_kernel(lib, rows, cols,
                                                                    staged_chunk, cluster,
                                                                    chunk, grid):
    # where the staged kernel's chunk fills under 0.8 of its threads' 1, 2, 4 or 8 vector
    # slots, the spread kernel takes the row: one buffer, the smallest cluster whose chunks
    # hold at most 7000 vectors (2 CTAs an SM in fp32), if they hold at least 4096
    need = -(-staged_chunk // 256)
    slots = 256 * next(n for n in (1, 2, 4, 8) if n >= need)
    assert staged_chunk / slots < 0.8
    p = camp.camp_layernorm_plan(X, W, BETA, Y, rows, cols, "f32")
    assert (p.kernel, p.vec_bytes, p.cluster, p.group, p.block, p.per_thread, p.grid) == \
        (camp.KERNEL_LAYERNORM_SPREAD, 16, cluster, chunk, 512, 1, grid)


def test_layernorm_staged_and_rows_thresholds(lib):
    p = camp.camp_layernorm_plan(X, W, BETA, Y, 4, 16384, "bf16")   # 2048 vectors: rows
    assert (p.kernel, p.group, p.per_thread) == (camp.KERNEL_LAYERNORM_ROWS, 512, 4)
    for rows, cols, nv in ((1025, 24576, 6), (2048, 24576, 6), (2048, 32768, 8)):   # rows
        p = camp.camp_layernorm_plan(X, W, BETA, Y, rows, cols, "bf16")
        assert (p.kernel, p.group, p.per_thread) == (camp.KERNEL_LAYERNORM_ROWS, 512, nv)


def test_layernorm_staged_plans_that_do_not_fit_are_refused(lib):
    # only refusals (an accepted plan would launch)
    for cols, dt, cl, stg in ((262144, camp.BF16, 8, 2),    # 4096 vectors a CTA
                              (131072, camp.BF16, 16, 5),   # 5 buffers are not built
                              (65536, camp.BF16, 3, 2)):    # cluster not a power of two
        plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_STAGED, vec_bytes=16, cluster=cl,
                         per_thread=stg)
        st = lib.camp_layernorm_with_plan(X, W, BETA, Y, 2, cols, ctypes.c_float(1e-5), dt,
                                          ctypes.byref(plan), None)
        assert st == camp.ERR_NOT_SUPPORTED, (cols, cl, stg)
    plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_STAGED, vec_bytes=16, cluster=4, per_thread=2)
    st = lib.camp_layernorm_with_plan(X, W, BETA + 2, Y, 2, 65536, ctypes.c_float(1e-5),
                                      camp.BF16, ctypes.byref(plan), None)
    assert st == camp.ERR_NOT_SUPPORTED   # beta not 16-byte aligned


@pytest.mark.parametrize("rows,cols,expect", [
    # at least 2 waves either way: more accesses per thread
    (65536, 2048, (64, 4, 16384)),
    (8192, 4096, (128, 4, 4096)),
    (8192, 2048, (64, 4, 2048)),
    (32768, 1024, (32, 4, 4096)),
])
def test_layernorm_many_waves_prefer_more_work_per_thread(lib, rows, cols, expect):
    p = camp.camp_layernorm_plan(X, W, BETA, Y, rows, cols, "bf16")
    assert (p.group, p.per_thread, p.grid) == expect
    q = camp.camp_rmsnorm_plan(X, W, Y, rows, cols, "bf16")
    assert q.per_thread <= p.per_thread


def test_layernorm_one_wave_test_uses_its_own_occupancy(lib):
    # RMSNorm's 64 x 4 holds 8 CTAs per SM, LayerNorm's 6 (it keeps more live): at 4096 x 2048
    # neither LayerNorm candidate fits one wave, so the one with fewer accesses per thread wins
    p = camp.camp_layernorm_plan(X, W, BETA, Y, 4096, 2048, "bf16")
    assert (p.group, p.per_thread, p.grid) == (128, 2, 2048)
    q = camp.camp_rmsnorm_plan(X, W, Y, 4096, 2048, "bf16")
    assert (q.group, q.per_thread, q.grid) == (64, 4, 1024)


def test_layernorm_rows_past_the_staged_kernel(lib):
    # the staged kernel holds up to 16 x 2048 sixteen-byte vectors (262144 bf16 / 131072
    # fp32 elements) and the element path of the rows kernel 1024 x 16 elements; wider rows
    # with 16-byte pitches take the spread kernel (16 CTAs of 512 threads, each CTA's chunk in
    # shared memory) while a chunk fits, everything else the wide kernel (one CTA of 1024
    # threads per row), any width
    for cols, dtype, b, kernel, vb, block in (
            (262152, "bf16", BETA, camp.KERNEL_LAYERNORM_SPREAD, 16, 512),
            (131076, "f32", BETA, camp.KERNEL_LAYERNORM_SPREAD, 16, 512),
            (524296, "f16", BETA, camp.KERNEL_LAYERNORM_SPREAD, 16, 512),
            (16385, "bf16", BETA + 2, camp.KERNEL_LAYERNORM_WIDE, 2, 1024),
            (300001, "bf16", BETA, camp.KERNEL_LAYERNORM_WIDE, 2, 1024),
            (2000000, "bf16", BETA, camp.KERNEL_LAYERNORM_WIDE, 16, 1024),
            (10**7 + 3, "f32", BETA, camp.KERNEL_LAYERNORM_WIDE, 4, 1024)):
        p = camp.camp_layernorm_plan(X, W, b, Y, 5, cols, dtype)
        assert (p.kernel, p.vec_bytes, p.block) == (kernel, vb, block), (cols, dtype)
        if kernel == camp.KERNEL_LAYERNORM_WIDE:
            assert (p.grid, p.cluster) == (5, 1)
        else:   # one buffer; 5 rows of 8 CTAs are split to 16 CTAs a row
            assert (p.per_thread, p.cluster, p.grid) == (1, 16, 80)


def test_layernorm_forced_wide_plans_that_do_not_fit_are_refused(lib):
    # the wide kernel takes 16-byte or element accesses, never wider than the pointers allow
    # (only refusals here: an accepted plan would launch)
    for vb, b in ((16, BETA + 2), (8, BETA), (4, BETA)):
        plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_WIDE, vec_bytes=vb)
        st = lib.camp_layernorm_with_plan(X, W, b, Y, 2, 4096, ctypes.c_float(1e-5), camp.BF16,
                                          ctypes.byref(plan), None)
        assert st == camp.ERR_NOT_SUPPORTED, (vb, b)


def test_layernorm_misaligned_beta_uses_element_accesses(lib):
    p = camp.camp_layernorm_plan(X, W, BETA + 2, Y, 4, 2048, "bf16")
    assert p.vec_bytes == 2
    p = camp.camp_layernorm_plan(X, W, BETA, Y, 4, 2048, "bf16")
    assert p.vec_bytes == 16


def test_layernorm_with_plan_checks_the_forced_plan(lib):
    bad = [
        camp.Plan(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=8, group=128, per_thread=2),
        camp.Plan(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=16, group=128, per_thread=1),
        camp.Plan(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=16, group=100, per_thread=4),
        camp.Plan(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=16, group=128, per_thread=5),
        camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=16, group=128, per_thread=2),
    ]
    for p in bad:
        st = lib.camp_layernorm_with_plan(X, W, BETA, Y, 4, 2048, ctypes.c_float(1e-5),
                                          camp.BF16, ctypes.byref(p), None)
        assert st == camp.ERR_NOT_SUPPORTED, (p.vec_bytes, p.group, p.per_thread)


def test_single_kernel_ops_refuse_a_plan_for_another_kernel(lib):
    p = camp.Plan(kernel=camp.KERNEL_ROPE, vec_bytes=16, per_thread=1)
    assert lib.camp_kv_rmsnorm_rope_cache_with_plan(
        X, W, SIN, COS, R_, Y, H_, 1, 4, 512, 64, 16, ctypes.c_float(1e-6), camp.BF16,
        ctypes.byref(p), None) == camp.ERR_NOT_SUPPORTED
    p = camp.Plan(kernel=camp.KERNEL_ROPE, vec_bytes=16, group=1)
    assert lib.camp_rope_interleaved_with_plan(X, SIN, COS, R_, Y, 4, 8, 64, 16, camp.BF16,
                                               ctypes.byref(p), None) == camp.ERR_NOT_SUPPORTED


# ------------------------------------------------------------------ KV concat + head repeat

CAT = [0x7C0000000000 + i * 0x1000000000 for i in range(5)]   # past, fresh, sin, cos, out


def _cat(lib, p, B=2, P=5, S=3, Hk=8, D=64, n_rep=4, dtype=camp.BF16):
    return lib.camp_kv_cat_repeat(*p, B, P, S, Hk, D, n_rep, dtype, None)


@pytest.mark.parametrize("change,kw,status", [
    ({}, {"dtype": 8}, camp.ERR_UNSUPPORTED_DTYPE),
    ({}, {"D": 7}, camp.ERR_INVALID_ARG),
    ({}, {"D": 0}, camp.ERR_INVALID_ARG),
    ({}, {"n_rep": 0}, camp.ERR_INVALID_ARG),
    ({}, {"P": -1}, camp.ERR_INVALID_ARG),
    ({}, {"Hk": -1}, camp.ERR_INVALID_ARG),
    ({0: None}, {}, camp.ERR_INVALID_ARG),                   # past needed when P > 0
    ({1: None}, {}, camp.ERR_INVALID_ARG),                   # fresh needed when S > 0
    ({4: None}, {}, camp.ERR_INVALID_ARG),
    ({2: None}, {}, camp.ERR_INVALID_ARG),                   # one table without the other
    ({3: None}, {}, camp.ERR_INVALID_ARG),
    ({2: CAT[2] + 2}, {}, camp.ERR_INVALID_ARG),             # table not fp32-aligned
    ({4: CAT[4] + 1}, {}, camp.ERR_INVALID_ARG),             # out not element-aligned
    ({4: CAT[0] + 64}, {}, camp.ERR_INVALID_ARG),            # out over past
    ({4: CAT[1]}, {}, camp.ERR_INVALID_ARG),                 # out over fresh (no in place)
    ({2: CAT[4] + 128}, {}, camp.ERR_INVALID_ARG),           # a table inside out
    ({}, {"Hk": 256, "D": 1024}, camp.ERR_NOT_SUPPORTED),    # a row needs more than one CTA
    ({}, {"B": 1 << 20, "P": 1 << 12, "Hk": 1, "D": 2}, camp.ERR_NOT_SUPPORTED),  # B*(P+S) >= 2^32
])
def test_kv_cat_argument_errors(lib, change, kw, status):
    p = list(CAT)
    for i, v in change.items():
        p[i] = v
    assert _cat(lib, p, **kw) == status


def test_kv_cat_empty_and_optional_pointers(lib):
    nil = [None] * 5
    for kw in ({"B": 0}, {"P": 0, "S": 0}, {"Hk": 0}):
        assert _cat(lib, nil, **kw) == camp.SUCCESS
    # P == 0: past may be NULL; S == 0: fresh and the tables may be NULL (planned only).
    p = camp.camp_kv_cat_repeat_plan(None, CAT[1], CAT[2], CAT[3], CAT[4], 1, 0, 16, 8, 64, 4,
                                     "bf16")
    assert p.kernel == camp.KERNEL_KV_CAT
    p = camp.camp_kv_cat_repeat_plan(CAT[0], None, None, None, CAT[4], 1, 16, 0, 8, 64, 4, "bf16")
    assert p.kernel == camp.KERNEL_KV_CAT
    # both tables NULL: copy the new rows
    p = camp.camp_kv_cat_repeat_plan(CAT[0], CAT[1], None, None, CAT[4], 1, 16, 4, 8, 64, 4, "f32")
    assert p.kernel == camp.KERNEL_KV_CAT


def test_kv_cat_plans(lib):
    # Llama-3.2-1B keys: 8 heads of 64, 4 query heads a key head. bf16: 4 vectors a half,
    # 2 heads a thread: 16 threads a row, 16 rows a CTA.
    p = camp.camp_kv_cat_repeat_plan(*CAT, 1, 4095, 1, 8, 64, 4, "bf16")
    assert (p.kernel, p.vec_bytes, p.group, p.block, p.grid) == (camp.KERNEL_KV_CAT, 16, 2, 256, 256)
    p = camp.camp_kv_cat_repeat_plan(*CAT, 2, 0, 4096, 8, 128, 4, "f32")
    assert (p.vec_bytes, p.group, p.grid) == (16, 2, 2 * 4096 // 4)   # 64 threads a row
    p = camp.camp_kv_cat_repeat_plan(*CAT, 1, 3, 4, 5, 6, 2, "bf16")     # odd heads, D/2 = 3
    assert (p.vec_bytes, p.group, p.grid) == (2, 1, 1)
    # fewer than 128 CTAs (256 rows: 16 with the bandwidth choice): the variant with the
    # smallest grid of at least 128
    p = camp.camp_kv_cat_repeat_plan(*CAT, 1, 255, 1, 8, 64, 4, "bf16")
    assert (p.vec_bytes, p.group, p.grid) == (4, 1, 128)
    p = camp.camp_kv_cat_repeat_plan(*CAT, 1, 3, 4, 64, 256, 2, "bf16")  # 64 heads of 256
    assert (p.vec_bytes, p.group) == (16, 4)                             # 16 x 16 threads
    p = camp.camp_kv_cat_repeat_plan(*CAT, 1, 3, 4, 128, 256, 2, "bf16")
    assert (p.vec_bytes, p.group) == (16, 8)
    # a misaligned input narrows the accesses of every tensor
    q = list(CAT)
    q[1] += 4
    p = camp.camp_kv_cat_repeat_plan(*q, 1, 3, 4, 8, 64, 4, "bf16")
    assert p.vec_bytes == 4


def test_kv_cat_with_plan_checks_the_forced_plan(lib):
    bad = [camp.Plan(kernel=camp.KERNEL_ROPE, vec_bytes=16, group=2),
           camp.Plan(kernel=camp.KERNEL_KV_CAT, vec_bytes=16, group=3),
           camp.Plan(kernel=camp.KERNEL_KV_CAT, vec_bytes=2, group=1),    # fp32 has no 2-byte
           camp.Plan(kernel=camp.KERNEL_KV_CAT, vec_bytes=16, group=1)]   # 3 floats a half
    for plan in bad:
        st = lib.camp_kv_cat_repeat_with_plan(*CAT, 1, 4, 4, 3, 6, 2, camp.F32,
                                              ctypes.byref(plan), None)
        assert st == camp.ERR_NOT_SUPPORTED, plan


# ------------------------------------------------------------------ staged RMSNorm plans

def _staged(cluster, stages):
    return camp.Plan(kernel=camp.KERNEL_RMSNORM_STAGED, vec_bytes=16, cluster=cluster,
                     per_thread=stages)


def test_staged_plans_that_do_not_fit_are_refused(lib):
    # Only refusals are checked here: an accepted plan would launch (the GPU tests run every
    # accepted variant on real memory). rows == 0 is a no-op whatever the plan.
    st = lib.camp_rmsnorm_with_plan(X, W, Y, 0, 131072, ctypes.c_float(1e-5), camp.BF16,
                                    ctypes.byref(_staged(8, 3)), None)
    assert st == camp.SUCCESS
    for (cols, dt, cl, stg) in [
        (131072, camp.BF16, 1, 2),      # a CTA chunk above 8 x 256 vectors
        (131072, camp.F32, 4, 3),       # 8192 vectors a CTA
        (65536, camp.F32, 8, 5),        # 5 buffers are not built
        (16384, camp.BF16, 3, 2),       # cluster not a power of two
        (16384, camp.BF16, 32, 2),      # cluster above 16
        (16384, camp.BF16, 2, 1),       # one buffer: no ring
        (16384, camp.BF16, 2, 5),       # more buffers than built
        (3001, camp.BF16, 1, 2),        # row pitch not a multiple of 16 bytes
    ]:
        st = lib.camp_rmsnorm_with_plan(X, W, Y, 2, cols, ctypes.c_float(1e-5), dt,
                                        ctypes.byref(_staged(cl, stg)), None)
        assert st == camp.ERR_NOT_SUPPORTED, (cols, cl, stg)


def test_staged_add_path_counts_both_staged_tensors(lib):
    R_ = 0x7F5000000000
    H_ = 0x7F6000000000
    # 32768 bf16 = 4096 vectors; x and r are both staged: 1 CTA would hold 4096 vectors
    # (above 8 x 256); 2 CTAs x 4 buffers need w + 8 x 32 KB, above the 224 KB budget
    for cl, stg in [(1, 2), (2, 4)]:
        st = lib.camp_add_rmsnorm_with_plan(X, R_, W, H_, Y, 2, 32768, ctypes.c_float(1e-5),
                                            camp.BF16, ctypes.byref(_staged(cl, stg)), None)
        assert st == camp.ERR_NOT_SUPPORTED, (cl, stg)


def test_staged_plan_needs_16_byte_accesses(lib):
    st = lib.camp_rmsnorm_with_plan(X + 2, W, Y, 2, 16384, ctypes.c_float(1e-5), camp.BF16,
                                    ctypes.byref(_staged(2, 2)), None)
    assert st == camp.ERR_NOT_SUPPORTED


def test_device_errors_argument_check(lib):
    assert lib.camp_device_errors(None, 0) == camp.ERR_INVALID_ARG


# ------------------------------------------------------------------ fp16 storage

def _fields(plan, dtype):
    """The plan's fields, or the status of a refused request."""
    try:
        p = plan(dtype)
    except camp.CampError as e:
        return e.status
    return (p.kernel, p.vec_bytes, p.group, p.per_thread, p.block, p.grid, p.cluster)


def _same(plan):
    assert _fields(plan, "f16") == _fields(plan, "bf16")


@pytest.mark.parametrize("shape", [(4096, 2048), (1, 8192), (64, 3001), (4096, 16384),
                                   (5, 65536), (256, 131072), (2, 262152), (3, 3000)])
def test_f16_plans_are_the_bf16_plans(lib, shape):
    """The planners look at the element size only: binary16 gets bf16's plans everywhere."""
    rows, cols = shape
    _same(lambda d: camp.camp_rmsnorm_plan(X, W, Y, rows, cols, d))
    _same(lambda d: camp.camp_add_rmsnorm_plan(X, R_, W, H_, Y, rows, cols, d))
    _same(lambda d: camp.camp_layernorm_plan(X, W, BETA, Y, rows, cols, d))


@pytest.mark.parametrize("B,S,H,D", [(1, 4096, 32, 64), (1, 8, 32, 64), (2, 3, 5, 6),
                                     (1, 65536, 32, 128), (1, 4, 1024, 256)])
def test_f16_rope_plans_are_the_bf16_plans(lib, B, S, H, D):
    _same(lambda d: camp.camp_rope_plan(X, SIN, COS, Y, B, S, H, D, d))
    _same(lambda d: camp.camp_rope_qk_plan(X, K_, SIN, COS, YQ, YK, B, S, H, 8, D, d))
    _same(lambda d: camp.camp_rope_interleaved_plan(*ILP, B * S, H, D, 16, d))
    _same(lambda d: camp.camp_kv_cat_repeat_plan(*CAT, B, S, S, 8, D, 4, d))


@pytest.mark.parametrize("Dn,Dr", [(512, 64), (128, 64), (100, 6)])
def test_f16_kv_cache_plans_are_the_bf16_plans(lib, Dn, Dr):
    _same(lambda d: camp.camp_kv_rmsnorm_rope_cache_plan(*KVP, 1, 4096, Dn, Dr, 8192, d))


def test_f16_dtype_names(lib):
    import torch
    for name in ("f16", "fp16", "float16", torch.float16, camp.F16):
        assert camp._dtype(name) == camp.F16 == 0


def test_wait_probe_refusals_launch_nothing(lib):
    # argument checks and plan refusals return before any launch (no device needed)
    plan_t = camp.Plan
    f = lib.camp_layernorm_wait_probe
    eps = ctypes.c_float(1e-5)
    for ns in (0, 999, 1_000_000_001):
        assert f(X, W, BETA, Y, 4, 65536, eps, camp.BF16, None, ns, None) == camp.ERR_INVALID_ARG
    # the rows kernel's width: no staged plan
    assert f(X, W, BETA, Y, 4, 2048, eps, camp.BF16, None, 100_000, None) == \
        camp.ERR_NOT_SUPPORTED
    for plan in (plan_t(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=16, group=512, per_thread=8),
                 plan_t(kernel=camp.KERNEL_LAYERNORM_WIDE, vec_bytes=16),
                 plan_t(kernel=camp.KERNEL_LAYERNORM_STAGED, vec_bytes=16, cluster=1, per_thread=2),
                 plan_t(kernel=camp.KERNEL_LAYERNORM_SPREAD, vec_bytes=16, cluster=3, per_thread=1),
                 plan_t(kernel=camp.KERNEL_RMSNORM_SPREAD, vec_bytes=16, cluster=2, per_thread=1)):
        assert f(X, W, BETA, Y, 4, 65536, eps, camp.BF16, ctypes.byref(plan), 100_000, None) == \
            camp.ERR_NOT_SUPPORTED, plan
    assert f(X, W, BETA, Y, 0, 65536, eps, camp.BF16, None, 100_000, None) == camp.SUCCESS


def test_rmsnorm_wait_probe_refusals_launch_nothing(lib):
    plan_t = camp.Plan
    f = lib.camp_rmsnorm_wait_probe
    eps = ctypes.c_float(1e-5)
    for ns in (0, 999, 1_000_000_001):
        assert f(X, W, Y, 4, 65536, eps, camp.BF16, None, ns, None) == camp.ERR_INVALID_ARG
    # 2048 vectors: the rows kernel's width, no staged plan
    assert f(X, W, Y, 4, 16384, eps, camp.BF16, None, 100_000, None) == camp.ERR_NOT_SUPPORTED
    for plan in (plan_t(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=16, group=512, per_thread=8),
                 plan_t(kernel=camp.KERNEL_RMSNORM_WIDE, vec_bytes=16),
                 plan_t(kernel=camp.KERNEL_RMSNORM_CLUSTER, vec_bytes=16, cluster=8, per_thread=8),
                 plan_t(kernel=camp.KERNEL_RMSNORM_STAGED, vec_bytes=16, cluster=1, per_thread=2),
                 plan_t(kernel=camp.KERNEL_RMSNORM_SPREAD, vec_bytes=16, cluster=3, per_thread=1),
                 plan_t(kernel=camp.KERNEL_LAYERNORM_SPREAD, vec_bytes=16, cluster=2, per_thread=1)):
        assert f(X, W, Y, 4, 65536, eps, camp.BF16, ctypes.byref(plan), 100_000, None) == \
            camp.ERR_NOT_SUPPORTED, plan
    assert f(X, W, Y, 0, 65536, eps, camp.BF16, None, 100_000, None) == camp.SUCCESS


@pytest.mark.parametrize("rows,cols,dtype,cluster,chunk,grid", [
    (256, 300000, "bf16", 16, 2344, 304),   # x and r staged: chunks of at most 3500 vectors
    (1024, 262152, "bf16", 16, 2049, 304),  # two CTAs an SM with the add
    (64, 524296, "bf16", 16, 4097, 144),    # 2 x 64 KB a CTA: one an SM
    (3, 131080, "f32", 16, 2049, 48),
])
def test_add_rmsnorm_rows_past_the_staged_kernel_take_the_spread_kernel(lib, rows, cols, dtype,
                                                                        cluster, chunk, grid):
    R, H = 0x7F3000000000, 0x7F4000000000
    p = camp.camp_add_rmsnorm_plan(X, R, W, H, Y, rows, cols, dtype)
    assert (p.kernel, p.vec_bytes, p.cluster, p.group, p.per_thread, p.block, p.grid) == \
        (camp.KERNEL_RMSNORM_SPREAD, 16, cluster, chunk, 1, 512, grid)
