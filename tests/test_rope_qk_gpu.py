"""Fused Q + K RoPE parity: camp_rope_qk (through the C ABI) against the fp64 oracle,
which rotates Q and K separately with the same tables. Tolerances as for camp_rope."""

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


def _check(x_cpu, sin_cpu, cos_cpu, y_dev, dtype, what):
    xs = inputs.to_numpy(x_cpu)
    got = inputs.to_numpy(y_dev).reshape(xs.shape)
    if dtype != "f32":
        assert_rounded_close(got, oracle.rope(xs, sin_cpu.numpy(), cos_cpu.numpy(), dtype),
                             dtype, what)
    else:
        assert_f32_close(got, oracle.rope_f64(xs.astype(np.float64), sin_cpu.numpy(),
                                              cos_cpu.numpy()), what)


def run_qk(B, S, Hq, Hk, D, dtype, seed=0, plan=None, inplace=False):
    q_cpu, sin_cpu, cos_cpu = inputs.rope_inputs(B, S, Hq, D, dtype, seed=seed)
    k_cpu, _, _ = inputs.rope_inputs(B, S, Hk, D, dtype, seed=seed + 1)
    q, k = q_cpu.cuda(), k_cpu.cuda()
    sn, cs = sin_cpu.cuda(), cos_cpu.cuda()
    yq, yk = (q, k) if inplace else (torch.empty_like(q), torch.empty_like(k))
    if plan is None:
        camp.camp_rope_qk(q, k, sn, cs, yq, yk, B, S, Hq, Hk, D, dtype)
    else:
        camp.camp_rope_qk_with_plan(q, k, sn, cs, yq, yk, B, S, Hq, Hk, D, dtype, plan)
    torch.cuda.synchronize()
    if Hq:
        _check(q_cpu, sin_cpu, cos_cpu, yq, dtype, f"rope_qk Q {dtype} {(B, S, Hq, D)}")
    if Hk:
        _check(k_cpu, sin_cpu, cos_cpu, yk, dtype, f"rope_qk K {dtype} {(B, S, Hk, D)}")


SHAPES = [(1, 4096, 32, 8, 64), (2, 33, 6, 2, 16), (1, 7, 3, 1, 64), (3, 17, 4, 4, 128),
          (2, 9, 5, 3, 6), (1, 5, 1024, 8, 256)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(shape, dtype):
    run_qk(*shape, dtype, seed=sum(shape))


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_fused_variant(dtype):
    es = ES[dtype]
    for vb in ((16, 8, 4, 2) if ES[dtype] == 2 else (16, 8, 4)):
        for hpt in (1, 2, 4, 8):
            D = 2 * (vb // es) * 3
            plan = camp.Plan(kernel=camp.KERNEL_ROPE, vec_bytes=vb, group=hpt)
            run_qk(2, 11, 2 * hpt + 1, hpt + 1, D, dtype, seed=vb * hpt, plan=plan)


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place(dtype):
    run_qk(2, 19, 8, 2, 64, dtype, seed=4, inplace=True)


@pytest.mark.parametrize("Hq,Hk", [(0, 8), (32, 0)])
def test_one_tensor_without_heads(Hq, Hk):
    run_qk(1, 64, Hq, Hk, 64, "bf16", seed=Hq + Hk)
