"""Interleaved RoPE with device position ids, and device table generation, against the
fp64 oracle (through the C ABI)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_memory_bound_gb300 import camp, inputs
from parity import DTYPES, ES, assert_f32_close, assert_rounded_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    torch.cuda.set_device(0)


def _f32_ulps(a, b):
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def run_case(T, H, D, dtype, max_pos=None, seed=0, plan=None, inplace=False):
    st = inputs.STORAGE[dtype]
    g = torch.Generator().manual_seed(seed)
    max_pos = max_pos or T + 7
    x_cpu = torch.randn(T, H, D, generator=g).to(st)
    sin_np, cos_np = inputs.rope_tables(max_pos, D, 10000.0)
    pos_cpu = torch.randint(0, max_pos, (T,), generator=g, dtype=torch.int32)
    if T > 3:
        pos_cpu[1] = -1
        pos_cpu[3] = max_pos
    y0_cpu = torch.randn(T, H, D, generator=g).to(st)
    x = x_cpu.cuda()
    y = x if inplace else y0_cpu.cuda()
    sn, cs, pos = torch.from_numpy(sin_np).cuda(), torch.from_numpy(cos_np).cuda(), pos_cpu.cuda()
    if plan is None:
        camp.camp_rope_interleaved(x, sn, cs, pos, y, T, H, D, max_pos, dtype)
    else:
        camp.camp_rope_interleaved_with_plan(x, sn, cs, pos, y, T, H, D, max_pos, dtype, plan)
    torch.cuda.synchronize()
    base = x_cpu if inplace else y0_cpu
    want = oracle.rope_interleaved(inputs.to_numpy(x_cpu), sin_np, cos_np, pos_cpu.numpy(),
                                   inputs.to_numpy(base), dtype)
    got = inputs.to_numpy(y)
    what = f"rope interleaved {dtype} {(T, H, D)}"
    if dtype != "f32":
        assert_rounded_close(got, want, dtype, what)
    else:
        # fp32: against the unrounded fp64 pair formula (written out here for the check)
        xs = inputs.to_numpy(x_cpu).astype(np.float64)
        ref = inputs.to_numpy(base).astype(np.float64).copy()
        p = pos_cpu.numpy()
        ok = (p >= 0) & (p < max_pos)
        c = cos_np[p[ok]].astype(np.float64)[:, None, :]
        s = sin_np[p[ok]].astype(np.float64)[:, None, :]
        x0, x1 = xs[ok][..., 0::2], xs[ok][..., 1::2]
        r = ref[ok]
        r[..., 0::2] = x0 * c - x1 * s
        r[..., 1::2] = x0 * s + x1 * c
        ref[ok] = r
        assert_f32_close(got, ref, what)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(1, 1, 2), (7, 3, 6), (33, 32, 64), (64, 8, 128), (300, 5, 20),
                                   (16, 64, 128), (2048, 32, 128)])
def test_shapes(shape, dtype):
    run_case(*shape, dtype, seed=sum(shape))


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_variant(dtype):
    es = ES[dtype]
    for vb in ((16, 8, 4) if ES[dtype] == 2 else (16, 8)):
        for hpt in (1, 2, 4, 8):
            D = 3 * vb // es                      # three vectors per head row
            plan = camp.Plan(kernel=camp.KERNEL_ROPE_INTERLEAVED, vec_bytes=vb, group=hpt)
            run_case(11, 2 * hpt + 1, D, dtype, seed=vb * hpt, plan=plan)


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place(dtype):
    run_case(40, 8, 64, dtype, seed=9, inplace=True)


@pytest.mark.parametrize("P,D,theta", [(4096, 64, 500000.0), (65536, 128, 500000.0),
                                       (1000, 6, 10000.0), (3, 2, 1e6)])
def test_device_tables(P, D, theta):
    s = torch.empty(P, D // 2, device="cuda")
    c = torch.empty(P, D // 2, device="cuda")
    camp.camp_rope_tables(s, c, P, D, theta)
    torch.cuda.synchronize()
    ws, wc = oracle.rope_tables(P, D, theta)
    # Both sides compute p * theta^(-2i/D) and sin/cos in fp64 and round once to fp32. Their
    # fp64 pow may differ by an ulp, which moves the angle by up to p * 2^-52 (1.5e-11 rad
    # at p = 65536); elsewhere that is far below an fp32 ulp, but near a zero of sin or cos
    # it can span a few tiny fp32 ulps. So each entry must be within 1 fp32 ulp or within
    # 1e-10 absolute.
    for got, want in ((s.cpu().numpy(), ws), (c.cpu().numpy(), wc)):
        close = (_f32_ulps(got, want) <= 1) | (np.abs(got.astype(np.float64) - want) <= 1e-10)
        assert close.all(), (np.argwhere(~close)[:5], got[~close][:5], want[~close][:5])
    np.testing.assert_array_equal(s[0].cpu().numpy(), 0.0)
    np.testing.assert_array_equal(c[0].cpu().numpy(), 1.0)
