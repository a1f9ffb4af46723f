"""Tensors past 2^32 elements (8.6 GB and more in bf16): the 64-bit offset arithmetic of the
kernels at the sizes where 32-bit math would wrap. Inputs are drawn on the device; rows
around every 2^31- and 2^32-element boundary and at both ends are copied back and checked
against the fp64 oracle (1 bf16 ulp, as everywhere)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_memory_bound_gb300 import camp, inputs
from parity import assert_bf16_close

import test_layernorm_gpu as ln_tests

pytestmark = pytest.mark.gpu

BIG = 1 << 32


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    torch.cuda.set_device(0)
    free, _ = torch.cuda.mem_get_info()
    if free < 60 * (1 << 30):
        pytest.skip("needs 60 GB of free device memory")
    yield
    torch.cuda.empty_cache()


def _sample_rows(n_rows: int, row_elems: int) -> list[int]:
    """Rows at both ends and around the element offsets 2^31, 2^32 and 2^33."""
    rows = {0, 1, n_rows - 2, n_rows - 1}
    for b in (1 << 31, 1 << 32, 1 << 33):
        r = b // row_elems
        rows.update(r + d for d in (-1, 0, 1))
    return sorted(r for r in rows if 0 <= r < n_rows)


def _randn_bf16(shape, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    flat = out.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):   # bounded fp32 temporaries
        n = min(step, flat.numel() - i)
        flat[i:i + n].copy_(torch.randn(n, generator=g, device="cuda"))
    return out


def test_rmsnorm_past_2_32_elements():
    rows, cols = (BIG // 4104) + 1000, 4104          # 4.3 G elements
    x = _randn_bf16((rows, cols), 1)
    w = (1 + 0.1 * torch.randn(cols, device="cuda")).to(torch.bfloat16)
    y = torch.empty_like(x)
    camp.camp_rmsnorm(x, w, y, rows, cols, 1e-5, "bf16")
    torch.cuda.synchronize()
    idx = torch.tensor(_sample_rows(rows, cols), device="cuda")
    want = oracle.rmsnorm(inputs.to_numpy(x[idx]), inputs.to_numpy(w), float(np.float32(1e-5)),
                          "bf16")
    assert_bf16_close(inputs.to_numpy(y[idx]), want, "rmsnorm past 2^32 elements")
    del x, y


def test_add_rmsnorm_past_2_32_elements():
    rows, cols = (BIG // 8192) + 77, 8192
    x = _randn_bf16((rows, cols), 2)
    r = _randn_bf16((rows, cols), 3)
    w = (1 + 0.1 * torch.randn(cols, device="cuda")).to(torch.bfloat16)
    h, y = torch.empty_like(x), torch.empty_like(x)
    camp.camp_add_rmsnorm(x, r, w, h, y, rows, cols, 1e-5, "bf16")
    torch.cuda.synchronize()
    idx = torch.tensor(_sample_rows(rows, cols), device="cuda")
    want_h, want_y = oracle.add_rmsnorm(inputs.to_numpy(x[idx]), inputs.to_numpy(r[idx]),
                                        inputs.to_numpy(w), float(np.float32(1e-5)), "bf16")
    np.testing.assert_array_equal(inputs.to_numpy(h[idx]), want_h)
    assert_bf16_close(inputs.to_numpy(y[idx]), want_y, "add_rmsnorm past 2^32 elements")
    del x, r, h, y


def test_layernorm_past_2_32_elements():
    rows, cols = (BIG // 2048) + 5, 2048
    x = _randn_bf16((rows, cols), 4)
    g = (1 + 0.1 * torch.randn(cols, device="cuda")).to(torch.bfloat16)
    b = torch.randn(cols, device="cuda").to(torch.bfloat16)
    y = torch.empty_like(x)
    camp.camp_layernorm(x, g, b, y, rows, cols, 1e-5, "bf16")
    torch.cuda.synchronize()
    idx = torch.tensor(_sample_rows(rows, cols), device="cuda")
    # LayerNorm's own tolerance (the fp32 error bound of its GPU tests)
    plan = camp.camp_layernorm_plan(x, g, b, y, rows, cols, "bf16")
    ln_tests.check(y[idx].cpu(), x[idx].cpu(), g.cpu(), b.cpu(), float(np.float32(1e-5)), plan,
                   "layernorm past 2^32 elements")
    del x, y


@pytest.mark.parametrize("cols,kinds", [
    (65536, (camp.KERNEL_RMSNORM_STAGED, camp.KERNEL_LAYERNORM_SPREAD)),   # rows in shared memory
    (262152, (camp.KERNEL_RMSNORM_SPREAD, camp.KERNEL_LAYERNORM_SPREAD)),  # a cluster per row
])
def test_wide_rows_past_2_32_elements(cols, kinds):
    rows = BIG // cols + 3
    x = _randn_bf16((rows, cols), 6)
    g = (1 + 0.1 * torch.randn(cols, device="cuda")).to(torch.bfloat16)
    b = torch.randn(cols, device="cuda").to(torch.bfloat16)
    y = torch.empty_like(x)
    idx = torch.tensor(_sample_rows(rows, cols), device="cuda")
    assert camp.camp_rmsnorm_plan(x, g, y, rows, cols, "bf16").kernel == kinds[0]
    camp.camp_rmsnorm(x, g, y, rows, cols, 1e-5, "bf16")
    torch.cuda.synchronize()
    want = oracle.rmsnorm(inputs.to_numpy(x[idx]), inputs.to_numpy(g), float(np.float32(1e-5)),
                          "bf16")
    assert_bf16_close(inputs.to_numpy(y[idx]), want, f"rmsnorm {rows}x{cols}")
    plan = camp.camp_layernorm_plan(x, g, b, y, rows, cols, "bf16")
    assert plan.kernel == kinds[1]
    camp.camp_layernorm(x, g, b, y, rows, cols, 1e-5, "bf16")
    torch.cuda.synchronize()
    ln_tests.check(y[idx].cpu(), x[idx].cpu(), g.cpu(), b.cpu(), float(np.float32(1e-5)), plan,
                   f"layernorm {rows}x{cols}")
    assert camp.camp_device_errors() == 0
    del x, y


def test_rope_qk_past_2_32_elements():
    S, Hq, Hk, D = (BIG // (40 * 64)) + 33, 32, 8, 64   # Q + K: 4.3 G elements
    q = _randn_bf16((1, S, Hq, D), 5)
    k = _randn_bf16((1, S, Hk, D), 6)
    sin_np, cos_np = inputs.rope_tables(S, D, 500000.0)
    sn, cs = torch.from_numpy(sin_np).cuda(), torch.from_numpy(cos_np).cuda()
    yq, yk = torch.empty_like(q), torch.empty_like(k)
    camp.camp_rope_qk(q, k, sn, cs, yq, yk, 1, S, Hq, Hk, D, "bf16")
    torch.cuda.synchronize()
    pos = _sample_rows(S, Hq * D)
    idx = torch.tensor(pos, device="cuda")
    for x, y, what in ((q, yq, "Q"), (k, yk, "K")):
        want = oracle.rope(inputs.to_numpy(x[:, idx]), sin_np[pos], cos_np[pos], "bf16")
        assert_bf16_close(inputs.to_numpy(y[:, idx]), want, f"rope {what} past 2^32 elements")
    del q, k, yq, yk


def test_kv_cat_repeat_past_2_32_elements():
    B, P, S, Hk, D, n_rep = 1, (BIG // (32 * 64)) + 100, 64, 8, 64, 4   # output 4.3 G elements
    past = _randn_bf16((B, P, Hk, D), 7)
    new = _randn_bf16((B, S, Hk, D), 8)
    sin_np, cos_np = inputs.rope_tables(P + S, D, 500000.0)
    sn, cs = torch.from_numpy(sin_np).cuda(), torch.from_numpy(cos_np).cuda()
    out = torch.empty(B, P + S, Hk * n_rep, D, dtype=torch.bfloat16, device="cuda")
    camp.camp_kv_cat_repeat(past, new, sn, cs, out, B, P, S, Hk, D, n_rep, "bf16")
    torch.cuda.synchronize()
    # cached rows: bit-exact copies, sampled around the output's 2^31 / 2^32 boundaries
    rows = [t for t in _sample_rows(P + S, Hk * n_rep * D) if t < P]
    idx = torch.tensor(rows, device="cuda")
    got = inputs.to_numpy(out[:, idx])
    want = np.repeat(inputs.to_numpy(past[:, idx]), n_rep, axis=2)
    np.testing.assert_array_equal(got, want)
    # the new rows: rotated at their absolute positions
    want_new = oracle.kv_cat_repeat(None, inputs.to_numpy(new), sin_np[P:], cos_np[P:], n_rep,
                                    "bf16")
    assert_bf16_close(inputs.to_numpy(out[:, P:]), want_new, "kv cat new rows past 2^32")
    del past, new, out
