"""Parity of the shared-memory-staged LayerNorm kernel (CAMP_KERNEL_LAYERNORM_STAGED) against
the fp64 oracle, through the C ABI: the default plan for wide rows, every (cluster, stages)
variant with forced plans, ragged chunks, CTAs with nothing but the row's head to load,
many rows per cluster; afterwards no bounded wait may have run out."""

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
    camp.camp_device_errors(clear=True)
    yield
    assert camp.camp_device_errors() == 0, "a bounded wait in a staged kernel ran out"


def plan(cluster: int, stages: int) -> camp.Plan:
    return camp.Plan(kernel=camp.KERNEL_LAYERNORM_STAGED, vec_bytes=16, cluster=cluster,
                     per_thread=stages)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [40000, 65536, 65544, 131072, 262144])
def test_wide_rows_default_plan(cols, dtype):
    if dtype == "f32" and cols > 131072:
        pytest.skip("past 16 x 2048 vectors: refused")
    ln_tests.run_case(6, cols, dtype, seed=cols % 97)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("stages", [2, 3, 4])
def test_every_variant(dtype, cluster, stages):
    e = 16 // ES[dtype]
    ln_tests.run_case(23, (cluster * 500 - 3) * e, dtype, seed=cluster * 10 + stages,
                      plan=plan(cluster, stages))


@pytest.mark.parametrize("dtype", DTYPES)
def test_ctas_with_only_the_head_to_load(dtype):
    e = 16 // ES[dtype]
    ln_tests.run_case(5, 3 * e, dtype, seed=1, plan=plan(16, 2))   # ranks 3..15 own nothing


@pytest.mark.parametrize("dtype", DTYPES)
def test_many_rows_per_cluster(dtype):
    cols = 65536 if ES[dtype] == 2 else 32768
    ln_tests.run_case(700, cols, dtype, seed=2)
    ln_tests.run_case(2000, 16384, dtype, seed=3, plan=plan(2, 3))


def test_in_place():
    ln_tests.run_case(40, 65536, "bf16", seed=4, in_place=True)
