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


def plan(cluster: int, stages: int, rows_per_step: int = 1) -> camp.Plan:
    return camp.Plan(kernel=camp.KERNEL_LAYERNORM_STAGED, vec_bytes=16, cluster=cluster,
                     per_thread=stages, rows_per_step=rows_per_step)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [40000, 65536, 65544, 131072, 262144])
def test_wide_rows_default_plan(cols, dtype):
    # fp32 rows past 131072 columns take the wide kernel (test_layernorm_wide_gpu.py)
    ln_tests.run_case(6, cols, dtype, seed=cols % 97)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("stages", [2, 3, 4])
@pytest.mark.parametrize("rps", [1, 2])
def test_every_variant(dtype, cluster, stages, rps):
    # 23 rows: with two rows a step every cluster's last step has one row
    e = 16 // ES[dtype]
    ln_tests.run_case(23, (cluster * 500 - 3) * e, dtype, seed=cluster * 10 + stages,
                      plan=plan(cluster, stages, rps))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rps,nvt", [(1, 1), (1, 2), (1, 4), (1, 8), (2, 1), (2, 2), (2, 4)])
def test_every_vectors_per_thread(dtype, rps, nvt):
    # chunks of just over (nvt - 1) * 256 vectors: the thread's last access is partly masked
    e = 16 // ES[dtype]
    cluster = 4
    chunk = (nvt - 1) * 256 + 7 if nvt > 1 else 200
    ln_tests.run_case(9, cluster * chunk * e, dtype, seed=rps * 10 + nvt,
                      plan=plan(cluster, 2 * rps, rps))


@pytest.mark.parametrize("dtype", DTYPES)
def test_ctas_with_only_the_head_to_load(dtype):
    e = 16 // ES[dtype]
    ln_tests.run_case(5, 3 * e, dtype, seed=1, plan=plan(16, 2))   # ranks 3..15 own nothing


@pytest.mark.parametrize("dtype", DTYPES)
def test_many_rows_per_cluster(dtype):
    cols = 65536 if ES[dtype] == 2 else 32768
    ln_tests.run_case(700, cols, dtype, seed=2)
    ln_tests.run_case(2000, 16384, dtype, seed=3, plan=plan(2, 3))


@pytest.mark.parametrize("dtype", DTYPES)
def test_gamma_beta_through_l1_with_short_chunks(dtype):
    # chunks of at most 4 vectors a thread stage gamma and beta in shared memory when that
    # leaves three CTAs an SM; with 4 buffers of 1000 vectors it does not, and they are read
    # through L1
    e = 16 // ES[dtype]
    for rps in (1, 2):
        ln_tests.run_case(11, 4 * 1000 * e, dtype, seed=rps, plan=plan(4, 4, rps))


@pytest.mark.parametrize("rps", [1, 2])
def test_in_place(rps):
    ln_tests.run_case(40, 65536, "bf16", seed=4, in_place=True, plan=plan(8, 4, rps))


@pytest.mark.parametrize("dtype", DTYPES)
def test_rows_far_from_their_shift(dtype):
    # the shift K = x[row, 0] 10 standard deviations from the mean, constant rows with one
    # different first element: the pairwise merges must keep the variance exact to fp32
    e = 16 // ES[dtype]
    cols = 8 * 1000 * e
    rows = 13
    for rps in (1, 2):
        ln_tests.run_case(rows, cols, dtype, seed=rps, plan=plan(8, 4, rps),
                          x_cpu=ln_tests._mixed_rows(rows, cols, dtype, rps))
