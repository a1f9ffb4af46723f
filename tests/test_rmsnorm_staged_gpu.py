"""Parity of the shared-memory-staged RMSNorm kernel (CAMP_KERNEL_RMSNORM_STAGED, plain and
fused residual add) against the fp64 oracle, through the C ABI with explicit plans: every
(cluster, stages) variant, ragged chunks, CTAs with nothing to load, many rows per cluster
(the buffer ring wraps several times), in-place calls; afterwards no bounded wait may have
run out (the library's device error word stays 0)."""

from __future__ import annotations

import pytest
import torch

from block_memory_bound_gb300 import camp
from parity import DTYPES, ES

import test_add_rmsnorm_gpu as add_tests
import test_rmsnorm_gpu as rms_tests

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
    return camp.Plan(kernel=camp.KERNEL_RMSNORM_STAGED, vec_bytes=16, cluster=cluster,
                     per_thread=stages)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("stages", [2, 3, 4])
def test_every_variant(dtype, cluster, stages):
    e = 16 // ES[dtype]
    # a ragged row (the last CTA's chunk is shorter), more rows than clusters
    cols = (cluster * 700 - 3) * e
    rms_tests.run_case(41, cols, dtype, seed=cluster * 10 + stages, plan=plan(cluster, stages))


@pytest.mark.parametrize("dtype", DTYPES)
def test_ctas_with_nothing_to_load(dtype):
    e = 16 // ES[dtype]
    # 5 vectors a row over 16 CTAs: ranks 5..15 own no vector
    rms_tests.run_case(7, 5 * e, dtype, seed=1, plan=plan(16, 2))
    rms_tests.run_case(3, e, dtype, seed=2, plan=plan(4, 3))


@pytest.mark.parametrize("dtype", DTYPES)
def test_many_rows_per_cluster(dtype):
    # far more rows than the device holds clusters: each cluster loops over many rows
    # (a CTA chunk holds at most 8 x 256 16-byte vectors)
    rms_tests.run_case(3000, 16384, dtype, seed=3, plan=plan(1 if ES[dtype] == 2 else 2, 3))
    rms_tests.run_case(777, 65536 if ES[dtype] == 2 else 32768, dtype, seed=4, plan=plan(4, 2))


@pytest.mark.parametrize("dtype", DTYPES)
def test_wide_rows(dtype):
    big = 262144 if ES[dtype] == 2 else 131072          # 16 CTAs of 2048 vectors
    rms_tests.run_case(64, big, dtype, seed=5, plan=plan(16, 2))
    ragged = 131072 + 8 if ES[dtype] == 2 else 65536 + 4  # 16 CTAs, the last one shorter
    rms_tests.run_case(33, ragged, dtype, seed=6, plan=plan(16, 3))


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place(dtype):
    rms_tests.run_case(50, 24576, dtype, seed=7, plan=plan(2 if ES[dtype] == 2 else 4, 3),
                       inplace=True)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cluster,stages", [(1, 2), (2, 3), (8, 4), (16, 2)])
def test_add_path(dtype, cluster, stages):
    e = 16 // ES[dtype]
    add_tests.run_case(37, (cluster * 600 - 5) * e, dtype, seed=cluster + stages,
                       plan=plan(cluster, stages))


@pytest.mark.parametrize("alias", ["h=r,y=x", "h=x,y=r"])
def test_add_path_in_place(alias):
    add_tests.run_case(29, 32768, "bf16", seed=9, plan=plan(2, 2), alias=alias)
