"""Parity of the wide LayerNorm kernel (CAMP_KERNEL_LAYERNORM_WIDE: one CTA per row,
block-stride sweeps, for rows no other kernel holds) against the fp64 oracle through the C
ABI, at the same bound as every LayerNorm variant: rows past the staged kernel's 262144
bf16 / 131072 fp32 columns, odd widths (element accesses), both access widths forced at
small sizes, rows whose shift lies far from the mean (the second pass), in place, more rows
than CTAs would need."""

from __future__ import annotations

import pytest
import torch

from block_memory_bound_gb300 import camp
from parity import DTYPES, ES

import test_layernorm_gpu as ln_tests

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [131076, 262152, 300001, 524296])
def test_rows_past_the_staged_kernel(cols, dtype):
    st = ln_tests.inputs.STORAGE[dtype]
    x = torch.empty(3, cols, device="cuda", dtype=st)
    g, b = (torch.empty(cols, device="cuda", dtype=st) for _ in range(2))
    # every one of these widths is past the staged kernel (or has an odd row pitch, which
    # leaves only element accesses) in all three storage types: the spread kernel while a
    # 16-byte-pitch row fits a cluster's shared memory, else the wide kernel
    p = camp.camp_layernorm_plan(x, g, b, x, 3, cols, dtype)
    assert p.kernel in (camp.KERNEL_LAYERNORM_WIDE, camp.KERNEL_LAYERNORM_SPREAD)
    ln_tests.run_case(3, cols, dtype, seed=cols % 89)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("vb", ["vector", "element"])
def test_forced_at_small_sizes(dtype, vb):
    es = ES[dtype]
    plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_WIDE, vec_bytes=16 if vb == "vector" else es)
    e = 16 // es
    for rows, cols in ((5, 1000 * e), (3, 8 * e), (2, 4096 * e + 8 * e)):
        ln_tests.run_case(rows, cols, dtype, seed=rows + cols, plan=plan)


@pytest.mark.parametrize("dtype", DTYPES)
def test_rows_far_from_their_shift(dtype):
    plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_WIDE, vec_bytes=16)
    e = 16 // ES[dtype]
    rows, cols = 9, 3000 * e
    ln_tests.run_case(rows, cols, dtype, seed=7, plan=plan,
                      x_cpu=ln_tests._mixed_rows(rows, cols, dtype, 7))


def test_in_place_and_many_rows():
    ln_tests.run_case(4, 300001, "bf16", seed=3, in_place=True)
    plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_WIDE, vec_bytes=16)
    ln_tests.run_case(400, 8192, "bf16", seed=4, plan=plan)
