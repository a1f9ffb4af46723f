"""LayerNorm parity: camp_layernorm (through the C ABI) against the fp64 oracle.

Tolerance, derived from the kernels' fp32 arithmetic (u = 2^-24), with one rounding count
k = K_ROUNDINGS for every compiled variant, so that no plan (and no later change of a
kernel's reduction) can widen it. The rows kernel's thread sums its L terms (accesses x
elements per access, at most 8 x 8) in two interleaved accumulators joined by one add (L/2
+ 1 roundings; L for one-element accesses), then a 5-level warp tree and at most 32 warp
partials: at most 64 + 5 + 32 = 101. The staged kernel's thread takes its own moments over
at most 64 elements (33 roundings a sum, one division), then merges them pairwise (Chan,
Golub and LeVeque: about 4 roundings a merge, relative to non-negative terms) over 5 warp
levels, 7 warps in turn and a 5-level butterfly over the cluster: about 33 + 4 x 17 + 1 =
102. K_ROUNDINGS = 128 covers both, and Higham's bound |fl(sum a) - sum a| <= k u sum |a|
applies to every sum. With K = x[row, 0],
c = mean|x - K| / sqrt(var + eps) (a property of the input row) and xhat the exact
normalized value, the fp32 kernel satisfies, per element,

    |y_kernel - y| <= u * ((k + 4) * |gamma| * (c + |xhat| * (1 + c)) + |y|)

(the deviation d = (x - K) - mu is off by <= (k + 3) u mean|x - K|; var by a relative
(k + 2) u + 2 (k + 3) u c; rsqrtf adds 2 ulp, var + eps and the product one rounding each,
and the final fma one rounding of |y|). A bf16 result adds the half ulp of its last
rounding, and an fp16 result the half ulp of binary16. LayerNorm has no 1-ulp rule like RMSNorm's: beta and gamma * xhat can cancel, and
then the fp32 error, relative to the operands, is many ulps of the tiny result.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_memory_bound_gb300 import camp, inputs
from parity import DTYPES, ES, half_ulp

pytestmark = pytest.mark.gpu

PAD = 64
U32 = 2.0 ** -24
K_ROUNDINGS = 128


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    torch.cuda.set_device(0)


def _decode(t: torch.Tensor) -> np.ndarray:
    return inputs.to_numpy(t.float()).astype(np.float64)


def _guarded(n, st):
    buf = torch.empty(n + 2 * PAD, dtype=st, device="cuda")
    buf.view(torch.int16 if st.itemsize == 2 else torch.int32).fill_(
        0x7FA5 if st.itemsize == 2 else 0x7FA5A5A5)
    return buf[PAD:PAD + n], buf


def _canaries_ok(buf, n):
    raw = buf.view(torch.int16 if buf.element_size() == 2 else torch.int32).cpu()
    sentinel = 0x7FA5 if buf.element_size() == 2 else 0x7FA5A5A5
    return bool((raw[:PAD] == sentinel).all()) and bool((raw[PAD + n:] == sentinel).all())


def check(got: torch.Tensor, x_cpu, g_cpu, b_cpu, eps32: float, plan: camp.Plan, what: str):
    rows, cols = x_cpu.shape
    dtype = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[x_cpu.dtype]
    del plan   # the bound is the same for every variant
    k = K_ROUNDINGS
    # In 16-bit storage the rows kernel takes the variance of a row in one pass,
    # sum((x - K)^2) / n - mu^2, whenever mu^2 <= 4 of that value; it then cancels at most
    # about 5 var against its inputs, so its error is at most about 14 times the summation
    # error, moving rstd by 7 k u relatively and y by 7 k u |xhat| |gamma|. The allowance
    # goes to the rows that can take that path (mu^2 <= 5 var in fp64: the kernel's fp32
    # test cannot move a row from beyond 5 to within 4), whatever the plan.
    one_pass = ES[dtype] == 2
    g, b = _decode(g_cpu), _decode(b_cpu)
    step = max(1, (1 << 22) // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        _check_rows(_decode(got[r0:r1]), _decode(x_cpu[r0:r1]), g, b, eps32, k, r0,
                    dtype, what, one_pass)


def _check_rows(y, x, g, b, eps32, k, r0, dtype, what, one_pass=False):
    ref, _ = oracle.layernorm_f64(x, g, b, eps32)
    dev = x - x[:, :1]
    var = ((x - x.mean(axis=1, keepdims=True)) ** 2).mean(axis=1, keepdims=True)
    sig = np.sqrt(var + eps32)
    c = np.abs(dev).mean(axis=1, keepdims=True) / sig
    xhat = (x - x.mean(axis=1, keepdims=True)) / sig
    bound = U32 * ((k + 4) * np.abs(g) * (c + np.abs(xhat) * (1 + c)) + np.abs(ref))
    if one_pass:
        mu = dev.mean(axis=1, keepdims=True)
        may = mu * mu <= 5.0 * var
        bound = bound + np.where(may, U32 * 8 * (k + 4) * np.abs(g) * np.abs(xhat), 0.0)
    if dtype != "f32":
        bound = bound + half_ulp(np.maximum(np.abs(ref), np.abs(y)), dtype)
    err = np.abs(y - ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements out of bound; first (row {r0 + i[0]}, "
            f"col {i[1]}): got "
            f"{y[tuple(i)]!r} want {ref[tuple(i)]!r} err {err[tuple(i)]:.3e} "
            f"bound {bound[tuple(i)]:.3e} (k={k})")


def run_case(rows, cols, dtype, eps=1e-5, seed=0, plan=None, in_place=False, x_cpu=None):
    x_rand, g_cpu, b_cpu = inputs.layernorm_inputs(rows, cols, dtype, seed=seed)
    if x_cpu is None:
        x_cpu = x_rand
    st = inputs.STORAGE[dtype]
    n = rows * cols
    x, g, b = x_cpu.cuda().contiguous(), g_cpu.cuda(), b_cpu.cuda()
    buf = None
    if in_place:
        y = x
    else:
        yf, buf = _guarded(n, st)
        y = yf.view(rows, cols)
    used = plan or camp.camp_layernorm_plan(x, g, b, y, rows, cols, dtype)
    if plan is None:
        camp.camp_layernorm(x, g, b, y, rows, cols, eps, dtype)
    else:
        camp.camp_layernorm_with_plan(x, g, b, y, rows, cols, eps, dtype, plan)
    torch.cuda.synchronize()
    eps32 = float(np.float32(eps))
    check(y.cpu().view(rows, cols), x_cpu, g_cpu, b_cpu, eps32, used,
          f"layernorm {dtype} {rows}x{cols}")
    if buf is not None:
        assert _canaries_ok(buf, n), "write outside the output"


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [1, 2, 7, 8, 64, 768, 1000, 2048, 3000, 3001, 4096, 8192,
                                  12288, 16384, 20000, 32768])
def test_shapes(cols, dtype):
    run_case(12, cols, dtype, seed=cols)


def test_widest_bf16_row():
    run_case(5, 65536, "bf16", seed=4)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [8, 2048, 3001, 20000])
def test_in_place(cols, dtype):
    run_case(7, cols, dtype, seed=cols + 1, in_place=True)


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_variant(dtype):
    es = ES[dtype]
    e = 16 // es
    for g in (32, 64, 128, 256, 512, 1024):
        for nv in (1, 2, 3, 4, 6, 8):
            plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=16, group=g,
                             per_thread=nv)
            run_case(3, max(e, (g * nv - 1) * e), dtype, seed=g + nv, plan=plan)
    for g in (32, 256, 1024):
        for nv in (1, 2, 4, 8, 16):
            plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=es, group=g,
                             per_thread=nv)
            run_case(3, max(1, g * nv - 1), dtype, seed=g * nv, plan=plan)


def _mixed_rows(rows: int, cols: int, dtype: str, seed: int) -> torch.Tensor:
    """Rows that take both variance paths of the rows kernel side by side in one CTA: N(0,1)
    rows (the shift within two standard deviations of the mean: one pass) alternating with
    rows whose first element (the shift K) lies 10 standard deviations out (mu^2 = 100 var:
    the second pass), and every fourth row a constant row with one different first element
    (x = [K, c, c, ...]: sum((x - K)^2) / n - mu^2 is within rounding of 0 and may come out
    negative in fp32, the other way to the second pass)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float64)
    for r in range(rows):
        if r % 4 == 1:
            x[r, 0] = x[r].mean() + 10.0 * x[r].std()
        elif r % 4 == 3:
            x[r, :] = 0.3 + 1e-3 * r
            x[r, 0] = 7.0
    return x.to(inputs.STORAGE[dtype])


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("group", [32, 64, 128, 256, 512, 1024])
def test_one_pass_and_second_pass_rows_in_one_cta(dtype, group):
    # Several rows a CTA where the group is smaller than 256 threads, several warps a row
    # from 64 threads up: the CTA-wide vote that sends a row group to the second pass must
    # not disturb the groups that skip it.
    e = 16 // ES[dtype]
    for nv in (2, 4):
        cols = group * nv * e - e   # the last access of the last thread masked
        plan = camp.Plan(kernel=camp.KERNEL_LAYERNORM_ROWS, vec_bytes=16, group=group,
                         per_thread=nv)
        rows = 4 * max(2, 256 // group) + 1
        run_case(rows, cols, dtype, seed=group + nv, plan=plan,
                 x_cpu=_mixed_rows(rows, cols, dtype, group * nv))


@pytest.mark.parametrize("dtype", DTYPES)
def test_constant_rows_give_beta_exactly(dtype):
    # every deviation is exactly 0 in both the kernel and the definition: y = beta
    rows, cols = 6, 3001
    st = inputs.STORAGE[dtype]
    _, g_cpu, b_cpu = inputs.layernorm_inputs(1, cols, dtype, seed=9)
    x_cpu = torch.tensor([0.0, 1.0, -3.5, 1000.0, 1e-3, 7.25]).to(st)[:, None].expand(rows, cols)
    x_cpu = x_cpu.contiguous()
    y = torch.empty(rows, cols, dtype=st, device="cuda")
    camp.camp_layernorm(x_cpu.cuda(), g_cpu.cuda(), b_cpu.cuda(), y, rows, cols, 1e-5, dtype)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), b_cpu[None, :].expand(rows, cols))


def test_zero_eps_constant_row_is_nan_like_the_definition():
    # var = 0 and eps = 0: (x - mean) / sqrt(var + eps) is 0 / 0
    rows, cols = 2, 100
    x = torch.full((rows, cols), 3.0, dtype=torch.float32)
    g = torch.ones(cols)
    b = torch.zeros(cols)
    y = torch.empty(rows, cols, device="cuda")
    camp.camp_layernorm(x.cuda(), g.cuda(), b.cuda(), y, rows, cols, 0.0, "f32")
    torch.cuda.synchronize()
    want = oracle.layernorm(x.numpy(), g.numpy(), b.numpy(), 0.0, "f32")
    assert np.isnan(want).all() and torch.isnan(y.cpu()).all()


def test_empty_rows_launch_nothing():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    camp.camp_layernorm(x, g, g.clone(), x, 0, 64, 1e-5, "bf16")


def test_tensor_convenience_matches_the_entry_point():
    x_cpu, g_cpu, b_cpu = inputs.layernorm_inputs(33, 1536, "bf16", seed=5)
    x, g, b = x_cpu.cuda(), g_cpu.cuda(), b_cpu.cuda()
    y1 = camp.layernorm(x.view(3, 11, 1536), g, b, eps=1e-6)
    y2 = torch.empty_like(x)
    camp.camp_layernorm(x, g, b, y2, 33, 1536, 1e-6, "bf16")
    torch.cuda.synchronize()
    assert torch.equal(y1.view(33, 1536), y2)


def test_config_bf16_4096x2048():
    run_case(4096, 2048, "bf16", seed=0)


def test_config_bf16_16384x8192():
    run_case(16384, 8192, "bf16", eps=1e-6, seed=0)


def test_config_f16_8192x4096():
    # the TileLang tutorial's example 2 (chapter 02): M = 8192 rows, H = 4096 columns, fp16
    run_case(8192, 4096, "f16", seed=0)
