"""RMSNorm parity: the CUDA path (through the C ABI) against the fp64 oracle.

Element-by-element at sizes the oracle finishes in seconds (several tiles and ragged
tails), at the full benchmark configurations, and on sampled rows at the largest sweep
sizes. bf16 and fp16 outputs must be within 1 ulp of the oracle rounded once; fp32 outputs within
1e-6 + 2e-6 |ref| of the oracle's fp64 result.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_memory_bound_gb300 import camp, inputs
from parity import DTYPES, ES, assert_bf16_close, assert_f32_close, assert_rounded_close

pytestmark = pytest.mark.gpu

PAD = 64   # canary elements on each side of every output


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()   # a missing library is a failure, not a skip
    torch.cuda.set_device(0)


def _guarded_empty(n: int, dtype: torch.dtype, offset: int = 0):
    """An output of n elements inside a canary-filled buffer; returns (view, buffer)."""
    buf = torch.empty(n + 2 * PAD + offset, dtype=dtype, device="cuda")
    if dtype.itemsize == 2:
        buf.view(torch.int16).fill_(0x7FA5)      # a NaN pattern (bf16 and fp16) no kernel produces
    else:
        buf.view(torch.int32).fill_(0x7FA5A5A5)
    return buf[PAD + offset:PAD + offset + n], buf


def _check_canaries(buf: torch.Tensor, n: int, offset: int = 0) -> None:
    raw = buf.view(torch.int16 if buf.element_size() == 2 else torch.int32).cpu()
    sentinel = 0x7FA5 if buf.element_size() == 2 else 0x7FA5A5A5
    head = raw[:PAD + offset]
    tail = raw[PAD + offset + n:]
    assert bool((head == sentinel).all()), "write before the output"
    assert bool((tail == sentinel).all()), "write past the output"


def _oracle_check(x_cpu, w_cpu, y_dev, eps: float, dtype: str, what: str) -> None:
    eps32 = float(np.float32(eps))
    xs = inputs.to_numpy(x_cpu).reshape(-1, x_cpu.shape[-1])
    ws = inputs.to_numpy(w_cpu)
    got = inputs.to_numpy(y_dev).reshape(xs.shape)
    if dtype != "f32":
        want = oracle.rmsnorm(xs, ws, eps32, dtype)
        assert_rounded_close(got, want, dtype, what)
    else:
        ref = oracle.rmsnorm_f64(xs.astype(np.float64), ws.astype(np.float64), eps32)
        assert_f32_close(got, ref, what)


def run_case(rows, cols, dtype, eps=1e-5, seed=0, stress=False, plan=None, inplace=False,
             x_offset=0, y_offset=0, x_cpu=None, w_cpu=None, stream=None):
    if x_cpu is None:
        x_cpu, w_cpu = inputs.rmsnorm_inputs(rows, cols, dtype, seed=seed, stress=stress)
    st = inputs.STORAGE[dtype]
    n = rows * cols
    xbuf = torch.empty(n + x_offset, dtype=st, device="cuda")
    x = xbuf[x_offset:x_offset + n].view(rows, cols)
    x.copy_(x_cpu.cuda())
    w = w_cpu.cuda()
    if inplace:
        y, ybuf = x, None
    else:
        yflat, ybuf = _guarded_empty(n, st, y_offset)
        y = yflat.view(rows, cols)
    if plan is None:
        camp.camp_rmsnorm(x, w, y, rows, cols, eps, dtype, stream)
    else:
        camp.camp_rmsnorm_with_plan(x, w, y, rows, cols, eps, dtype, plan, stream)
    torch.cuda.synchronize()
    _oracle_check(x_cpu, w_cpu, y, eps, dtype, f"rmsnorm {dtype} {rows}x{cols}")
    if ybuf is not None:
        _check_canaries(ybuf, n, y_offset)
    return y


# ------------------------------------------------------------------ shapes and tails

COLS = [1, 2, 7, 8, 33, 64, 256, 1000, 2048, 2056, 3000, 3001, 4096, 8192, 8200, 20000]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("rows", [1, 3, 37])
def test_shapes_and_tails(rows, cols, dtype):
    run_case(rows, cols, dtype, seed=rows * 7 + cols)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [12288, 16384, 40000, 65536, 70000, 131072, 262144, 300001,
                                  524296])
def test_wide_rows(cols, dtype):
    run_case(3, cols, dtype, seed=cols)


def test_cluster_rows_many():
    run_case(777, 16384, "bf16", seed=9)


@pytest.mark.parametrize("dtype", DTYPES)
def test_many_rows_ragged(dtype):
    run_case(1001, 3000, dtype, seed=5)


def test_p3_style_deterministic_case():
    # xserv unit-test style data: 4 rows of 768, x = ((i mod 17) - 8) / 10, gamma 0.5/0.7/0.9.
    for dtype in DTYPES:
        x_cpu, w_cpu = inputs.p3_style_rmsnorm_inputs(4, 768, dtype)
        run_case(4, 768, dtype, x_cpu=x_cpu, w_cpu=w_cpu)


@pytest.mark.parametrize("eps", [0.0, 1e-6, 1e-5, 1e-2])
def test_eps_values(eps):
    run_case(17, 2048, "bf16", eps=eps, seed=11)
    run_case(17, 2048, "f16", eps=eps, seed=13)
    run_case(17, 2048, "f32", eps=eps, seed=12)


def test_constant_rows_match_closed_form_within_tolerance():
    # x_j = c: y_j = w_j * sign(c) / sqrt(1 + eps/c^2); checked through the oracle rule.
    cols = 2048
    x_cpu = torch.tensor([1.0, -2.0, 0.01, 300.0], dtype=torch.float32)[:, None].expand(4, cols)
    x_cpu = x_cpu.contiguous().to(torch.bfloat16)
    _, w_cpu = inputs.rmsnorm_inputs(1, cols, "bf16", seed=3)
    run_case(4, cols, "bf16", x_cpu=x_cpu, w_cpu=w_cpu)


# ------------------------------------------------------------------ every compiled variant

def _variants(dtype: str):
    es = ES[dtype]
    out = []
    for g in (32, 64, 128, 256, 512, 1024):
        for nv in (1, 2, 3, 4, 6, 8):
            out.append((16, g, nv))
    for g in (32, 256, 1024):
        for nv in (1, 2, 4, 8, 16):
            out.append((es, g, nv))
    return out


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_rows_variant(dtype):
    es = ES[dtype]
    for vb, g, nv in _variants(dtype):
        e = vb // es
        # Widest row the variant holds, minus one vector: the last accesses are masked.
        cols = max(e, (g * nv - 1) * e) if g * nv > 1 else e
        plan = camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=vb, group=g, per_thread=nv)
        run_case(5, cols, dtype, seed=g + nv, plan=plan)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cluster", [2, 4, 8, 16])
def test_every_cluster_variant(dtype, cluster):
    e = 16 // ES[dtype]
    for nv in (1, 2, 3, 4, 6, 8):
        # one vector short of the capacity: the last CTA's last access is masked
        cols = (cluster * 256 * nv - 1) * e
        plan = camp.Plan(kernel=camp.KERNEL_RMSNORM_CLUSTER, vec_bytes=16, per_thread=nv,
                         cluster=cluster)
        run_case(3, cols, dtype, seed=cluster * 10 + nv, plan=plan)
    # rows far shorter than the cluster: most CTAs have nothing to load
    plan = camp.Plan(kernel=camp.KERNEL_RMSNORM_CLUSTER, vec_bytes=16, per_thread=1,
                     cluster=cluster)
    run_case(4, 8 * e, dtype, seed=cluster, plan=plan)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("vb", ["vector", "element"])
def test_wide_kernel_forced(dtype, vb):
    es = ES[dtype]
    plan = camp.Plan(kernel=camp.KERNEL_RMSNORM_WIDE, vec_bytes=16 if vb == "vector" else es)
    run_case(9, 8192, dtype, seed=2, plan=plan)
    run_case(4, 24, dtype, seed=3, plan=plan)


# ------------------------------------------------------------------ aliasing, alignment, streams

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [2048, 3001, 40000, 70000, 524296])
def test_in_place(cols, dtype):
    run_case(7, cols, dtype, seed=cols + 1, inplace=True)


@pytest.mark.parametrize("dtype", DTYPES)
def test_misaligned_pointers_take_the_element_path(dtype):
    x_cpu, w_cpu = inputs.rmsnorm_inputs(9, 2048, dtype, seed=4)
    x = torch.empty(9 * 2048 + 1, dtype=inputs.STORAGE[dtype], device="cuda")[1:].view(9, 2048)
    w = w_cpu.cuda()
    plan = camp.camp_rmsnorm_plan(x, w, torch.empty_like(x), 9, 2048, dtype)
    assert plan.vec_bytes == (2 if ES[dtype] == 2 else 4)
    run_case(9, 2048, dtype, x_offset=1, y_offset=1, x_cpu=x_cpu, w_cpu=w_cpu)


def test_side_stream():
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run_case(64, 2048, "bf16", seed=8, stream=s)


def test_empty_rows_is_a_no_op():
    y, ybuf = _guarded_empty(16, torch.bfloat16)
    camp.camp_rmsnorm(0, 0, 0, 0, 16, 1e-5, "bf16")
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    camp.camp_rmsnorm(x, x, y, 0, 16, 1e-5, "bf16")
    torch.cuda.synchronize()
    _check_canaries(ybuf, 16)


# ------------------------------------------------------------------ benchmark configurations

def test_config_fp32_64x2048():
    run_case(64, 2048, "f32", eps=1e-5, seed=0)


def test_config_bf16_4096x2048():
    run_case(4096, 2048, "bf16", eps=1e-5, seed=0)


def test_config_bf16_16384x8192_stress():
    run_case(16384, 8192, "bf16", eps=1e-6, seed=0, stress=True)


def test_f16_stress_rows_partly_subnormal():
    # binary16: the stress recipe's 1e-4 rows hold subnormal inputs, its 1e3 rows reach ~4e3
    run_case(1000, 4096, "f16", eps=1e-6, seed=21, stress=True)


def test_f16_overflow_rounds_to_infinity():
    # One nonzero element a row: y = x / sqrt(x^2 / 64 + eps) * w, about 8 * 10000 in
    # magnitude, past binary16's largest finite value (65504): +inf and -inf, as in the oracle.
    cols = 64
    x = torch.zeros(2, cols)
    x[0, 0] = 1.0
    x[1, 5] = -3.0
    w = torch.full((cols,), 10000.0)
    y = run_case(2, cols, "f16", x_cpu=x.to(torch.float16), w_cpu=w.to(torch.float16)).cpu()
    assert y[0, 0].item() == float("inf") and y[1, 5].item() == float("-inf")
    assert int(torch.isinf(y).sum()) == 2


def _sampled_rows(rows: int, k: int, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    idx = torch.randperm(rows, generator=g)[:k]
    return torch.unique(torch.cat([idx, torch.tensor([0, rows - 1])]))


@pytest.mark.parametrize("tokens", [1, 8, 64, 512, 4096, 65536])
@pytest.mark.parametrize("hidden", [2048, 3000, 8192])
def test_sweep_device_inputs_sampled(tokens, hidden):
    # The benchmark's own inputs (drawn on the device) and launch; the oracle checks a
    # sample of whole rows (all rows when there are few).
    x, w = inputs.rmsnorm_inputs(tokens, hidden, "bf16", seed=0, device="cuda")
    y = torch.empty_like(x)
    camp.camp_rmsnorm(x, w, y, tokens, hidden, 1e-5, "bf16")
    torch.cuda.synchronize()
    idx = _sampled_rows(tokens, 512, seed=tokens + hidden).cuda()
    xs = inputs.to_numpy(x[idx])
    ws = inputs.to_numpy(w)
    want = oracle.rmsnorm(xs, ws, float(np.float32(1e-5)), "bf16")
    assert_bf16_close(inputs.to_numpy(y[idx]), want, f"sweep {tokens}x{hidden}")
    del x, y
    torch.cuda.empty_cache()
