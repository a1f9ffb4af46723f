"""Parity of the spread kernels (CAMP_KERNEL_RMSNORM_SPREAD, CAMP_KERNEL_LAYERNORM_SPREAD: a
cluster of CTAs per row, each holding its whole chunk of the row in shared memory) against
the fp64 oracle through the C ABI, at the RMSNorm rule (1 ulp / 1e-6 + 2e-6 |ref|) and the
LayerNorm bound: every cluster size and buffer count forced at small sizes with ragged
chunks and ranks that own nothing, more rows than resident clusters, LayerNorm rows that
take the second pass, in place, and the default plan for rows past the staged kernel;
afterwards no bounded wait may have run out."""

from __future__ import annotations

import pytest
import torch

from block_memory_bound_gb300 import camp
from parity import DTYPES, ES

import test_add_rmsnorm_gpu as add_tests
import test_layernorm_gpu as ln_tests
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
    assert camp.camp_device_errors() == 0, "a bounded wait in a spread kernel ran out"


def rms_plan(cluster, stages):
    return camp.Plan(kernel=camp.KERNEL_RMSNORM_SPREAD, vec_bytes=16, cluster=cluster,
                     per_thread=stages)


def ln_plan(cluster, stages):
    return camp.Plan(kernel=camp.KERNEL_LAYERNORM_SPREAD, vec_bytes=16, cluster=cluster,
                     per_thread=stages)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("stages", [1, 2, 3])
def test_every_variant(dtype, cluster, stages):
    # chunks that are not a multiple of the 512 threads, the last rank's chunk short
    e = 16 // ES[dtype]
    cols = (cluster * 1300 - 7) * e
    rms_tests.run_case(9, cols, dtype, seed=cluster + stages, plan=rms_plan(cluster, stages))
    ln_tests.run_case(9, cols, dtype, seed=cluster * stages, plan=ln_plan(cluster, stages))


@pytest.mark.parametrize("dtype", DTYPES)
def test_ranks_with_nothing_to_load(dtype):
    e = 16 // ES[dtype]
    rms_tests.run_case(5, 3 * e, dtype, seed=1, plan=rms_plan(16, 2))
    ln_tests.run_case(5, 3 * e, dtype, seed=1, plan=ln_plan(16, 2))


@pytest.mark.parametrize("dtype", DTYPES)
def test_many_rows_per_cluster(dtype):
    # more rows than the clusters the device holds at once: each cluster loops, through the
    # ring's phases more than once
    e = 16 // ES[dtype]
    rms_tests.run_case(301, 16 * 900 * e, dtype, seed=2, plan=rms_plan(16, 2))
    ln_tests.run_case(301, 16 * 900 * e, dtype, seed=2, plan=ln_plan(16, 2))


@pytest.mark.parametrize("dtype", DTYPES)
def test_layernorm_rows_far_from_their_shift(dtype):
    e = 16 // ES[dtype]
    rows, cols = 13, 8 * 1000 * e
    for stages in (1, 2):
        ln_tests.run_case(rows, cols, dtype, seed=stages, plan=ln_plan(8, stages),
                          x_cpu=ln_tests._mixed_rows(rows, cols, dtype, stages))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("plan", [None, (8, 1), (16, 2)])
def test_rmsnorm_stress_rows(plan, dtype):
    # the stress distribution (1% of rows x1e3, 1% x1e-4; in fp16 partly subnormal) on rows
    # past the staged kernel: fp32 sums over a row spread across the cluster's CTAs
    p = None if plan is None else rms_plan(*plan)
    cols = 262152 if ES[dtype] == 2 else 131076
    rms_tests.run_case(200, cols, dtype, eps=1e-6, seed=4, stress=True, plan=p)


def test_rmsnorm_constant_rows_match_closed_form_within_tolerance():
    # x_j = c: y_j = w_j * sign(c) / sqrt(1 + eps/c^2), and a zero row gives 0 (eps > 0)
    cols = 262152
    vals = torch.tensor([1.0, -2.0, 0.01, 300.0, 0.0], dtype=torch.float32)
    x_cpu = vals[:, None].expand(5, cols).contiguous().to(torch.bfloat16)
    _, w_cpu = rms_tests.inputs.rmsnorm_inputs(1, cols, "bf16", seed=3)
    y = rms_tests.run_case(5, cols, "bf16", x_cpu=x_cpu, w_cpu=w_cpu)
    assert bool((y[4] == 0).all())


def test_in_place():
    rms_tests.run_case(21, 16 * 2100 * 8, "bf16", seed=3, plan=rms_plan(16, 2), inplace=True)
    ln_tests.run_case(21, 16 * 2100 * 8, "bf16", seed=3, plan=ln_plan(16, 2), in_place=True)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [262152, 524296, 1048576])
def test_default_plan_past_the_staged_kernel(cols, dtype):
    st = ln_tests.inputs.STORAGE[dtype]
    x = torch.empty(3, cols, device="cuda", dtype=st)
    w, b = (torch.empty(cols, device="cuda", dtype=st) for _ in range(2))
    # the spread kernel while one buffer of a 16th of the row fits 224 KB (fp32 at 1048576
    # columns does not: the two-sweep kernels)
    spread = (cols * ES[dtype] // 16 + 15) // 16 * 16 + 16 <= 224 * 1024
    assert (camp.camp_rmsnorm_plan(x, w, x, 3, cols, dtype).kernel ==
            (camp.KERNEL_RMSNORM_SPREAD if spread else camp.KERNEL_RMSNORM_WIDE))
    assert (camp.camp_layernorm_plan(x, w, b, x, 3, cols, dtype).kernel ==
            (camp.KERNEL_LAYERNORM_SPREAD if spread else camp.KERNEL_LAYERNORM_WIDE))
    del x, w, b
    rms_tests.run_case(3, cols, dtype, seed=cols % 13)
    ln_tests.run_case(3, cols, dtype, seed=cols % 17)


@pytest.mark.parametrize("kind,rows,cols,dtype,plan", [
    # more rows than one round of the resident clusters, not a whole number of rounds: the
    # last round's rows on a part of the clusters
    ("ln", 256, 131072, "bf16", None),       # 4-CTA clusters, 28 rows in the last round
    ("rms", 60, 300000, "bf16", None),       # 8-CTA clusters, 9 rows in the last round
    ("ln", 300, 140000, "f32", None),        # two CTAs an SM
    ("rms", 200, 140000, "f16", None),
    ("ln", 403, 140000, "bf16", "4x2"),      # two buffers
    ("rms", 501, 65536, "bf16", "2x1"),
])
def test_rows_past_a_round_of_clusters(kind, rows, cols, dtype, plan):
    p = None
    if plan is not None:
        cl, st = map(int, plan.split("x"))
        p = ln_plan(cl, st) if kind == "ln" else rms_plan(cl, st)
    if kind == "ln":
        ln_tests.run_case(rows, cols, dtype, seed=rows % 11, plan=p)
    else:
        rms_tests.run_case(rows, cols, dtype, seed=rows % 11, plan=p)


# ------------------------------------------------------------------ the residual add

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("stages", [1, 2])
def test_add_every_variant(dtype, cluster, stages):
    # x and r staged, h stored from the statistics sweep and formed again for the output
    e = 16 // ES[dtype]
    add_tests.run_case(7, (cluster * 1300 - 7) * e, dtype, seed=cluster + stages,
                       plan=rms_plan(cluster, stages))


@pytest.mark.parametrize("alias", ["h=r,y=x", "h=x,y=r"])
def test_add_in_place(alias):
    add_tests.run_case(21, 16 * 2100 * 8, "bf16", seed=5, plan=rms_plan(16, 2), alias=alias)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,cols", [(3, 262152), (300, 280000)])
def test_add_default_plan_past_the_staged_kernel(rows, cols, dtype):
    # the planner's spread plan for the add path (its choice is pinned by the host tests)
    add_tests.run_case(rows, cols, dtype, seed=cols % 7)


def test_forced_plans_that_do_not_fit_are_refused():
    x = torch.zeros(2, 4096, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    for cl, st in ((3, 2), (16, 4), (16, 0), (32, 1)):
        with pytest.raises(camp.CampError) as ei:
            camp.camp_rmsnorm_with_plan(x, w, y, 2, 4096, 1e-5, "bf16", rms_plan(cl, st))
        assert ei.value.status == camp.ERR_NOT_SUPPORTED
    # 2 buffers of a 262 KB chunk do not fit shared memory
    big = torch.zeros(1, 16 * 16400 * 8, dtype=torch.bfloat16, device="cuda")
    wb = torch.ones(16 * 16400 * 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(camp.CampError) as ei:
        camp.camp_rmsnorm_with_plan(big, wb, torch.empty_like(big), 1, 16 * 16400 * 8, 1e-5,
                                    "bf16", rms_plan(16, 2))
    assert ei.value.status == camp.ERR_NOT_SUPPORTED
