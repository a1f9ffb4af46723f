"""KV concatenation + grouped-query head repeat parity: camp_kv_cat_repeat (through the C
ABI) against the fp64 oracle. Copied rows (the cache, and the new rows when no tables are
given) must be bit-exact; rotated rows follow the RoPE tolerances. Canary regions around
the output must be left as they were."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_memory_bound_gb300 import camp, inputs
from parity import DTYPES, ES, assert_f32_close, assert_rounded_close

pytestmark = pytest.mark.gpu

THETA = 500000.0
CANARY = 4096   # elements on each side of the output


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    torch.cuda.set_device(0)


def _offset_copy(t_cpu: torch.Tensor, elems: int) -> tuple[torch.Tensor, torch.Tensor]:
    """A device copy of t that starts `elems` elements into a larger buffer (misaligns it)."""
    buf = torch.empty(t_cpu.numel() + elems, dtype=t_cpu.dtype, device="cuda")
    view = buf[elems:].view(t_cpu.shape)
    view.copy_(t_cpu)
    return buf, view


def run_case(B, P, S, Hk, D, n_rep, dtype, seed=0, plan=None, tables=True, shift=0):
    st = inputs.STORAGE[dtype]
    g = torch.Generator().manual_seed(seed)
    T = P + S
    past_cpu = torch.randn(B, P, Hk, D, generator=g).to(st)
    new_cpu = torch.randn(B, S, Hk, D, generator=g).to(st)
    sin_np, cos_np = inputs.rope_tables(max(T, 1), D, THETA)
    keep = []
    past = new = None
    if P > 0:
        buf, past = _offset_copy(past_cpu, shift)
        keep.append(buf)
    if S > 0:
        buf, new = _offset_copy(new_cpu, shift)
        keep.append(buf)
    sn = torch.from_numpy(sin_np).cuda() if tables else None
    cs = torch.from_numpy(cos_np).cuda() if tables else None
    n_out = B * T * Hk * n_rep * D
    canary_cpu = torch.randn(2 * CANARY + n_out, generator=g).to(st)
    out_buf = canary_cpu.cuda()
    out = out_buf[CANARY:CANARY + n_out]
    if plan is None:
        camp.camp_kv_cat_repeat(past, new, sn, cs, out, B, P, S, Hk, D, n_rep, dtype)
    else:
        camp.camp_kv_cat_repeat_with_plan(past, new, sn, cs, out, B, P, S, Hk, D, n_rep, dtype,
                                          plan)
    torch.cuda.synchronize()
    what = f"kv cat {dtype} {(B, P, S, Hk, D, n_rep)} tables={tables}"
    got_buf = inputs.to_numpy(out_buf)
    want_buf = inputs.to_numpy(canary_cpu)
    np.testing.assert_array_equal(got_buf[:CANARY], want_buf[:CANARY], what + " (canary)")
    np.testing.assert_array_equal(got_buf[CANARY + n_out:], want_buf[CANARY + n_out:],
                                  what + " (canary)")
    got = got_buf[CANARY:CANARY + n_out].reshape(B, T, Hk * n_rep, D)

    want = oracle.kv_cat_repeat(inputs.to_numpy(past_cpu) if P else None,
                                inputs.to_numpy(new_cpu), sin_np[:T] if tables else None,
                                cos_np[:T] if tables else None, n_rep, dtype)
    # Copied rows: bit for bit.
    copied = T if not tables else P
    np.testing.assert_array_equal(got[:, :copied], want[:, :copied], what + " (copied rows)")
    if not tables or S == 0:
        return
    if dtype != "f32":
        assert_rounded_close(got[:, P:], want[:, P:], dtype, what)
    else:
        # fp32: against the unrounded fp64 rotation at table rows P .. P+S-1, repeated
        ref = oracle.rope_f64(inputs.to_numpy(new_cpu), sin_np[P:T], cos_np[P:T])
        ref = np.repeat(ref, n_rep, axis=2)
        assert_f32_close(got[:, P:], ref, what)


# Llama-3.2-1B keys (8 heads of 64, 32 query heads): prefill, decode with a long cache and a
# chunked prefill; ragged head counts and widths; S = 0 and P = 0; n_rep = 1.
SHAPES = [
    (1, 0, 256, 8, 64, 4), (1, 511, 1, 8, 64, 4), (2, 300, 45, 8, 64, 4),
    (2, 37, 5, 3, 6, 2), (3, 5, 0, 2, 8, 3), (1, 0, 7, 5, 10, 1), (1, 1, 1, 1, 2, 1),
    (1, 64, 64, 8, 128, 4), (4, 17, 13, 2, 128, 7), (1, 9, 3, 64, 256, 2),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(shape, dtype):
    run_case(*shape, dtype, seed=sum(shape))


@pytest.mark.parametrize("dtype", DTYPES)
def test_without_tables_is_a_copy(dtype):
    run_case(2, 40, 24, 8, 64, 4, dtype, seed=3, tables=False)


@pytest.mark.parametrize("dtype", DTYPES)
def test_element_aligned_pointers(dtype):
    # inputs one element past a 16-byte boundary: element accesses
    run_case(2, 33, 9, 8, 64, 4, dtype, seed=5, shift=1)


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_variant(dtype):
    es = ES[dtype]
    for vb in ((16, 8, 4, 2) if ES[dtype] == 2 else (16, 8, 4)):
        for hpt in (1, 2, 4, 8):
            D = 2 * 3 * vb // es                      # three vectors a half
            plan = camp.Plan(kernel=camp.KERNEL_KV_CAT, vec_bytes=vb, group=hpt)
            run_case(2, 7, 6, 2 * hpt + 1, D, 3, dtype, seed=vb * hpt, plan=plan)


def test_full_size_decode_and_prefill():
    # Llama-3.2-1B shapes at the benchmark's size: a 4096-position cache with a 512-token
    # chunk, and a 4096-token prefill.
    run_case(1, 3584, 512, 8, 64, 4, "bf16", seed=11)
    run_case(1, 0, 4096, 8, 64, 4, "bf16", seed=12)
