"""The failure path of the staged and spread kernels' bounded waits, exercised without
faulting anything: camp_layernorm_wait_probe runs the staged or spread LayerNorm with every
mbarrier wait bounded by a short limit and each CTA's first row copy left unissued, so every
CTA's first wait runs out. The kernel must return (the call completes), set the timeout bit in the
device error word, store nothing, and leave the library usable: the bit reads back once and
clears, and the next normal call is clean and correct."""

from __future__ import annotations

import pytest
import torch

from block_memory_bound_gb300 import camp

import test_layernorm_gpu as ln_tests

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    torch.cuda.set_device(0)
    camp.camp_device_errors(clear=True)


def staged(cluster, rows_per_step=1):
    return camp.Plan(kernel=camp.KERNEL_LAYERNORM_STAGED, vec_bytes=16, cluster=cluster,
                     per_thread=2, rows_per_step=rows_per_step)


def spread(cluster, stages=1):
    return camp.Plan(kernel=camp.KERNEL_LAYERNORM_SPREAD, vec_bytes=16, cluster=cluster,
                     per_thread=stages)


@pytest.mark.parametrize("dtype,rows,cols,plan", [
    ("bf16", 6, 65536, None),            # the staged plan for these arguments
    ("bf16", 6, 65536, staged(4)),
    ("f32", 5, 65536, staged(8)),
    ("f16", 40, 131072, staged(8)),
    ("f32", 7, 32768, staged(8, 2)),     # two rows a step
    ("bf16", 6, 65536, spread(2)),
    ("f16", 40, 131072, spread(4)),
    ("f32", 5, 300000, spread(16)),      # the second pass and its exchange on every row
    ("bf16", 400, 40000, spread(1, 2)),  # 2-3 rows a CTA: the second buffer's copy lands
])
def test_a_wait_that_runs_out_sets_the_bit_and_stores_nothing(dtype, rows, cols, plan):
    x = torch.randn(rows, cols, device="cuda").to(ln_tests.inputs.STORAGE[dtype])
    g = torch.ones(cols, device="cuda", dtype=x.dtype)
    b = torch.zeros(cols, device="cuda", dtype=x.dtype)
    yflat, buf = ln_tests._guarded(rows * cols, x.dtype)
    bits = torch.int16 if buf.element_size() == 2 else torch.int32   # the canary is a NaN
    before = buf.view(bits).clone()
    assert camp.camp_device_errors(clear=True) == 0
    camp.camp_layernorm_wait_probe(x, g, b, yflat, rows, cols, 1e-5, dtype, wait_ns=200_000,
                                   plan=plan)
    torch.cuda.synchronize()
    assert camp.camp_device_errors() & camp.DEVICE_ERROR_WAIT_TIMEOUT
    assert torch.equal(buf.view(bits), before), "a CTA whose wait ran out stored output"
    # the bit reads back until cleared, then stays clear
    assert camp.camp_device_errors(clear=True) & camp.DEVICE_ERROR_WAIT_TIMEOUT
    assert camp.camp_device_errors() == 0
    # the next normal call is clean and correct
    ln_tests.run_case(rows, cols, dtype, seed=rows)
    assert camp.camp_device_errors() == 0


def test_probe_argument_checks():
    x = torch.zeros(4, 65536, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(65536, device="cuda", dtype=torch.bfloat16)
    y = torch.empty_like(x)
    for ns in (0, 999, 1_000_000_001):
        with pytest.raises(camp.CampError) as ei:
            camp.camp_layernorm_wait_probe(x, g, g, y, 4, 65536, 1e-5, "bf16", wait_ns=ns)
        assert ei.value.status == camp.ERR_INVALID_ARG
    small = torch.zeros(4, 2048, device="cuda", dtype=torch.bfloat16)   # the rows kernel
    with pytest.raises(camp.CampError) as ei:
        camp.camp_layernorm_wait_probe(small, g, g, torch.empty_like(small), 4, 2048, 1e-5,
                                       "bf16", wait_ns=100_000)
    assert ei.value.status == camp.ERR_NOT_SUPPORTED
    for plan in (camp.Plan(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=16, group=512,
                           per_thread=8),          # a kernel without bounded waits
                 camp.Plan(kernel=camp.KERNEL_LAYERNORM_WIDE, vec_bytes=16),
                 staged(1),                        # 8192 vectors do not fit one CTA
                 spread(3)):                       # not a power of two
        with pytest.raises(camp.CampError) as ei:
            camp.camp_layernorm_wait_probe(x, g, g, y, 4, 65536, 1e-5, "bf16", wait_ns=100_000,
                                           plan=plan)
        assert ei.value.status == camp.ERR_NOT_SUPPORTED
    assert camp.camp_device_errors() == 0


# ------------------------------------------------------------------ RMSNorm

import test_rmsnorm_gpu as rms_tests   # noqa: E402  (the RMSNorm run-and-compare helper)


def rms_staged(cluster, stages):
    return camp.Plan(kernel=camp.KERNEL_RMSNORM_STAGED, vec_bytes=16, cluster=cluster,
                     per_thread=stages)


def rms_spread(cluster, stages=1):
    return camp.Plan(kernel=camp.KERNEL_RMSNORM_SPREAD, vec_bytes=16, cluster=cluster,
                     per_thread=stages)


@pytest.mark.parametrize("dtype,rows,cols,plan", [
    ("bf16", 6, 65536, None),              # the staged plan for these arguments
    ("f32", 5, 65536, rms_staged(16, 2)),
    ("f16", 40, 131072, rms_staged(16, 3)),
    ("bf16", 700, 65536, rms_staged(8, 3)),  # a dozen rows a cluster after the failed one
    ("bf16", 6, 300000, rms_spread(8)),      # a copy group a warp
    ("f32", 5, 262144, rms_spread(16)),
    ("bf16", 400, 140000, rms_spread(4, 2)),  # two buffers, about ten rows a cluster
])
def test_an_rmsnorm_wait_that_runs_out_sets_the_bit_and_stores_nothing(dtype, rows, cols,
                                                                        plan):
    x = torch.randn(rows, cols, device="cuda").to(ln_tests.inputs.STORAGE[dtype])
    w = torch.ones(cols, device="cuda", dtype=x.dtype)
    yflat, buf = ln_tests._guarded(rows * cols, x.dtype)
    bits = torch.int16 if buf.element_size() == 2 else torch.int32   # the canary is a NaN
    before = buf.view(bits).clone()
    assert camp.camp_device_errors(clear=True) == 0
    camp.camp_rmsnorm_wait_probe(x, w, yflat, rows, cols, 1e-5, dtype, wait_ns=200_000,
                                 plan=plan)
    torch.cuda.synchronize()
    assert camp.camp_device_errors() & camp.DEVICE_ERROR_WAIT_TIMEOUT
    assert torch.equal(buf.view(bits), before), "a CTA whose wait ran out stored output"
    assert camp.camp_device_errors(clear=True) & camp.DEVICE_ERROR_WAIT_TIMEOUT
    assert camp.camp_device_errors() == 0
    rms_tests.run_case(rows, cols, dtype, seed=rows)   # the next normal call
    assert camp.camp_device_errors() == 0
