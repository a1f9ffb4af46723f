"""Rotate-half RoPE parity: the CUDA path (through the C ABI) against the fp64 oracle.

bf16 and fp16 outputs must be within 1 ulp of the oracle rounded once; fp32 outputs within
1e-6 + 2e-6 |ref| of the oracle's fp64 result. Position 0 (cos = 1, sin = 0) must
reproduce the input bit for bit.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_memory_bound_gb300 import camp, inputs
from parity import DTYPES, ES, assert_bf16_close, assert_f32_close, assert_rounded_close

pytestmark = pytest.mark.gpu

PAD = 64


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    torch.cuda.set_device(0)


def _oracle_check(x_cpu, sin_cpu, cos_cpu, y_dev, dtype, what):
    xs = inputs.to_numpy(x_cpu)
    got = inputs.to_numpy(y_dev).reshape(xs.shape)
    s = sin_cpu.numpy()
    c = cos_cpu.numpy()
    if dtype != "f32":
        assert_rounded_close(got, oracle.rope(xs, s, c, dtype), dtype, what)
    else:
        assert_f32_close(got, oracle.rope_f64(xs.astype(np.float64), s, c), what)


def run_case(B, S, H, D, dtype, seed=0, plan=None, inplace=False, x_offset=0, y_offset=0,
             table_offset=0, theta=500000.0):
    x_cpu, sin_cpu, cos_cpu = inputs.rope_inputs(B, S, H, D, dtype, seed=seed, theta=theta)
    st = inputs.STORAGE[dtype]
    n = B * S * H * D
    xbuf = torch.empty(n + x_offset, dtype=st, device="cuda")
    x = xbuf[x_offset:].view(B, S, H, D)
    x.copy_(x_cpu.cuda())
    nt = S * (D // 2)
    tbuf = torch.empty(2 * (nt + table_offset), dtype=torch.float32, device="cuda")
    sin_d = tbuf[table_offset:table_offset + nt].view(S, D // 2)
    cos_d = tbuf[nt + 2 * table_offset:].view(S, D // 2)
    sin_d.copy_(sin_cpu.cuda())
    cos_d.copy_(cos_cpu.cuda())
    if inplace:
        y, ybuf = x, None
    else:
        ybuf = torch.empty(n + 2 * PAD + y_offset, dtype=st, device="cuda")
        ybuf.view(torch.int16 if st.itemsize == 2 else torch.int32).fill_(
            0x7FA5 if st.itemsize == 2 else 0x7FA5A5A5)
        y = ybuf[PAD + y_offset:PAD + y_offset + n].view(B, S, H, D)
    if plan is None:
        camp.camp_rope(x, sin_d, cos_d, y, B, S, H, D, dtype)
    else:
        camp.camp_rope_with_plan(x, sin_d, cos_d, y, B, S, H, D, dtype, plan)
    torch.cuda.synchronize()
    _oracle_check(x_cpu, sin_cpu, cos_cpu, y, dtype, f"rope {dtype} {(B, S, H, D)}")
    if ybuf is not None:
        raw = ybuf.view(torch.int16 if st.itemsize == 2 else torch.int32).cpu()
        sentinel = 0x7FA5 if st.itemsize == 2 else 0x7FA5A5A5
        assert bool((raw[:PAD + y_offset] == sentinel).all()), "write before the output"
        assert bool((raw[PAD + y_offset + n:] == sentinel).all()), "write past the output"
    return x_cpu, y


SHAPES = [(1, 1, 1, 2), (2, 3, 5, 6), (1, 7, 32, 64), (1, 16, 8, 128), (2, 33, 3, 20),
          (3, 5, 7, 136), (1, 9, 4, 16), (2, 4, 6, 32), (1, 300, 32, 64), (4, 64, 8, 128)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(shape, dtype):
    run_case(*shape, dtype, seed=sum(shape))


@pytest.mark.parametrize("dtype", DTYPES)
def test_position_zero_is_identity(dtype):
    x_cpu, y = run_case(2, 5, 8, 64, dtype, seed=1)
    got = inputs.to_numpy(y)[:, 0]
    np.testing.assert_array_equal(got, inputs.to_numpy(x_cpu)[:, 0])


@pytest.mark.parametrize("kernel", ["tiled", "flat"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_every_variant(dtype, kernel):
    es = ES[dtype]
    vbs = (16, 8, 4, 2) if ES[dtype] == 2 else (16, 8, 4)
    kid = camp.KERNEL_ROPE if kernel == "tiled" else camp.KERNEL_ROPE_FLAT
    for vb in vbs:
        for hpt in (1, 2, 4, 8):
            e = vb // es
            D = 2 * e * 3                       # three vectors per half
            H = 2 * hpt + 1                     # a ragged last head group
            plan = camp.Plan(kernel=kid, vec_bytes=vb, group=hpt)
            run_case(2, 5, H, D, dtype, seed=vb + hpt, plan=plan)
            run_case(3, 37, H, D, dtype, seed=vb + hpt + 1, plan=plan)


@pytest.mark.parametrize("S", [1, 2, 3, 7, 33, 1000, 4097, 70001])
def test_table_row_of_every_position(S):
    # B > 1 makes the flattened position b*S + s wrap around S; the table row is derived
    # on the device by a multiply-shift division.
    run_case(3, S, 2, 16, "bf16", seed=S)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(1, 8, 32, 64), (2, 3, 5, 6)])
def test_in_place(shape, dtype):
    run_case(*shape, dtype, seed=3, inplace=True)


@pytest.mark.parametrize("dtype", DTYPES)
def test_misaligned_pointers(dtype):
    run_case(1, 6, 4, 64, dtype, seed=5, x_offset=1, y_offset=1, table_offset=1)


def test_empty_is_a_no_op():
    camp.camp_rope(0, 0, 0, 0, 0, 4, 2, 8, "bf16")
    camp.camp_rope(0, 0, 0, 0, 1, 0, 2, 8, "bf16")
    camp.camp_rope(0, 0, 0, 0, 1, 4, 0, 8, "bf16")
    torch.cuda.synchronize()


def test_config_q_1x4096x32x64():
    run_case(1, 4096, 32, 64, "bf16", seed=0)


def test_config_k_1x4096x8x64():
    run_case(1, 4096, 8, 64, "bf16", seed=0)


def test_config_f16_1x4096x32x128():
    # the TileLang tutorial's exercise E13 (chapter 02): B = 1, 32 heads, S = 4096, d = 128, fp16
    run_case(1, 4096, 32, 128, "f16", seed=0)


@pytest.mark.parametrize("tokens", [1, 8, 64, 512, 4096, 65536])
@pytest.mark.parametrize("H,D", [(32, 64), (8, 64), (32, 128), (8, 128)])
def test_sweep_device_inputs_sampled(tokens, H, D):
    # The benchmark's own inputs (drawn on the device) and launch; the oracle checks all
    # heads of a sample of positions.
    x, sin_d, cos_d = inputs.rope_inputs(1, tokens, H, D, "bf16", seed=0, device="cuda")
    y = torch.empty_like(x)
    camp.camp_rope(x, sin_d, cos_d, y, 1, tokens, H, D, "bf16")
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(tokens * 31 + H + D)
    pos = torch.unique(torch.cat([torch.randperm(tokens, generator=g)[:256],
                                  torch.tensor([0, tokens - 1])]))
    xs = inputs.to_numpy(x[:, pos.cuda()])
    ss = sin_d[pos.cuda()].cpu().numpy()
    cs = cos_d[pos.cuda()].cpu().numpy()
    want = oracle.rope(xs, ss, cs, "bf16")
    assert_bf16_close(inputs.to_numpy(y[:, pos.cuda()]), want, f"rope sweep {tokens}x{H}x{D}")
    del x, y
    torch.cuda.empty_cache()
