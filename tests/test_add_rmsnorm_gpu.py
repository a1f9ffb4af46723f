"""Fused residual add + RMSNorm parity: camp_add_rmsnorm (through the C ABI) against the
fp64 oracle. h = x + r must match the oracle's once-rounded sum (within 1 bf16 ulp /
the fp32 rule, and in practice bit for bit); y = RMSNorm(h) * w within the RMSNorm rule."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_memory_bound_gb300 import camp, inputs
from parity import DTYPES, ES, assert_f32_close, assert_rounded_close

pytestmark = pytest.mark.gpu

PAD = 64


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    torch.cuda.set_device(0)


def _guarded(n, st):
    buf = torch.empty(n + 2 * PAD, dtype=st, device="cuda")
    buf.view(torch.int16 if st.itemsize == 2 else torch.int32).fill_(
        0x7FA5 if st.itemsize == 2 else 0x7FA5A5A5)
    return buf[PAD:PAD + n], buf


def _canaries_ok(buf, n):
    raw = buf.view(torch.int16 if buf.element_size() == 2 else torch.int32).cpu()
    sentinel = 0x7FA5 if buf.element_size() == 2 else 0x7FA5A5A5
    return bool((raw[:PAD] == sentinel).all()) and bool((raw[PAD + n:] == sentinel).all())


def run_case(rows, cols, dtype, eps=1e-5, seed=0, plan=None, alias=None):
    """alias: None (separate outputs), "h=r,y=x" or "h=x,y=r" (in place)."""
    x_cpu, w_cpu = inputs.rmsnorm_inputs(rows, cols, dtype, seed=seed)
    r_cpu, _ = inputs.rmsnorm_inputs(rows, cols, dtype, seed=seed + 1, stress=True)
    st = inputs.STORAGE[dtype]
    n = rows * cols
    x, r, w = x_cpu.cuda().contiguous(), r_cpu.cuda().contiguous(), w_cpu.cuda()
    bufs = []
    if alias == "h=r,y=x":
        h, y = r, x
    elif alias == "h=x,y=r":
        h, y = x, r
    else:
        hf, hb = _guarded(n, st)
        yf, yb = _guarded(n, st)
        h, y = hf.view(rows, cols), yf.view(rows, cols)
        bufs = [hb, yb]
    if plan is None:
        camp.camp_add_rmsnorm(x, r, w, h, y, rows, cols, eps, dtype)
    else:
        camp.camp_add_rmsnorm_with_plan(x, r, w, h, y, rows, cols, eps, dtype, plan)
    torch.cuda.synchronize()
    xs, rs, ws = (inputs.to_numpy(t) for t in (x_cpu, r_cpu, w_cpu))
    eps32 = float(np.float32(eps))
    want_h, want_y = oracle.add_rmsnorm(xs, rs, ws, eps32, dtype)
    got_h = inputs.to_numpy(h).reshape(rows, cols)
    got_y = inputs.to_numpy(y).reshape(rows, cols)
    what = f"add_rmsnorm {dtype} {rows}x{cols}"
    if dtype != "f32":
        np.testing.assert_array_equal(got_h, want_h, err_msg=what + " h")
        assert_rounded_close(got_y, want_y, dtype, what + " y")
    else:
        np.testing.assert_array_equal(got_h, want_h, err_msg=what + " h")
        ref = oracle.rmsnorm_f64(want_h.astype(np.float64), ws.astype(np.float64), eps32)
        assert_f32_close(got_y, ref, what + " y")
    for b in bufs:
        assert _canaries_ok(b, n), "write outside an output"


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [1, 7, 8, 64, 1000, 2048, 3000, 3001, 8192, 20000, 40000,
                                  70000, 300001])
def test_shapes(cols, dtype):
    run_case(3, cols, dtype, seed=cols)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("alias", ["h=r,y=x", "h=x,y=r"])
@pytest.mark.parametrize("cols", [2048, 3001, 40000, 300001])
def test_in_place(cols, dtype, alias):
    run_case(5, cols, dtype, seed=cols + 3, alias=alias)


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_variant(dtype):
    es = ES[dtype]
    e = 16 // es
    for g in (32, 64, 128, 256, 512, 1024):
        for nv in (1, 2, 3, 4, 6, 8):
            if g == 1024 and nv == 8:
                continue   # not built on the add path
            plan = camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=16, group=g,
                             per_thread=nv)
            run_case(3, max(e, (g * nv - 1) * e), dtype, seed=g + nv, plan=plan)
    for g in (32, 256, 1024):
        for nv in (1, 2, 4, 8, 16):
            plan = camp.Plan(kernel=camp.KERNEL_RMSNORM_ROWS, vec_bytes=es, group=g,
                             per_thread=nv)
            run_case(3, max(1, g * nv - 1), dtype, seed=g * nv, plan=plan)
    for cl in (2, 4, 8, 16):
        for nv in (1, 3, 8):
            plan = camp.Plan(kernel=camp.KERNEL_RMSNORM_CLUSTER, vec_bytes=16, per_thread=nv,
                             cluster=cl)
            run_case(2, (cl * 256 * nv - 1) * e, dtype, seed=cl * nv, plan=plan)
    for vb in (16, es):
        plan = camp.Plan(kernel=camp.KERNEL_RMSNORM_WIDE, vec_bytes=vb)
        run_case(4, 8192, dtype, seed=vb, plan=plan)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,cols", [(777, 12288), (153, 16384), (9, 24576), (1, 32768)])
def test_default_plans_past_1024_vectors(rows, cols, dtype):
    # 1024-thread groups on the 16-bit types (2, 2, 3 and 4 accesses a thread), the
    # staged kernel for fp32 at 24576 columns and more
    run_case(rows, cols, dtype, seed=rows + cols)


def test_config_bf16_4096x2048():
    run_case(4096, 2048, "bf16", seed=0)


def test_config_bf16_16384x8192():
    run_case(16384, 8192, "bf16", eps=1e-6, seed=0)
