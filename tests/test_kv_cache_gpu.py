"""KV RMSNorm + RoPE + cache scatter parity: camp_kv_rmsnorm_rope_cache (through the C ABI)
against the fp64 oracle. Written cache rows follow the RMSNorm / RoPE rules; rows no token
names, and tokens with a padding slot, must leave the caches bit for bit as they were."""

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


def run_case(B, S, Dn, Dr, dtype, seed=0, plan=None, num_slots=None, pad=True):
    st = inputs.STORAGE[dtype]
    g = torch.Generator().manual_seed(seed)
    kv_cpu = torch.randn(B, S, Dn + Dr, generator=g).to(st)
    gamma_cpu = (1 + 0.1 * torch.randn(Dn, generator=g)).to(st)
    _, sin_cpu, cos_cpu = inputs.rope_inputs(1, S, 1, Dr, dtype, seed=seed)
    ns = num_slots or 2 * B * S + 3
    slots_cpu = torch.randperm(ns, generator=g)[:B * S].to(torch.int64)
    if pad and B * S > 2:
        slots_cpu[1] = -1
        slots_cpu[-1] = ns + 5
    cn_cpu = torch.randn(ns, Dn, generator=g).to(st)
    cr_cpu = torch.randn(ns, Dr, generator=g).to(st)
    kv, gamma, sn, cs = kv_cpu.cuda(), gamma_cpu.cuda(), sin_cpu.cuda(), cos_cpu.cuda()
    slots, cn, cr = slots_cpu.cuda(), cn_cpu.cuda(), cr_cpu.cuda()
    if plan is None:
        camp.camp_kv_rmsnorm_rope_cache(kv, gamma, sn, cs, slots, cn, cr, B, S, Dn, Dr, ns,
                                        1e-5, dtype)
    else:
        camp.camp_kv_rmsnorm_rope_cache_with_plan(kv, gamma, sn, cs, slots, cn, cr, B, S, Dn,
                                                  Dr, ns, 1e-5, dtype, plan)
    torch.cuda.synchronize()
    want_n, want_r = oracle.kv_rmsnorm_rope_cache(
        inputs.to_numpy(kv_cpu), inputs.to_numpy(gamma_cpu), sin_cpu.numpy(), cos_cpu.numpy(),
        slots_cpu.numpy(), inputs.to_numpy(cn_cpu), inputs.to_numpy(cr_cpu), Dn,
        float(np.float32(1e-5)), dtype)
    got_n, got_r = inputs.to_numpy(cn), inputs.to_numpy(cr)
    s_np = slots_cpu.numpy()
    written = np.zeros(ns, bool)
    written[s_np[(s_np >= 0) & (s_np < ns)]] = True
    what = f"kv cache {dtype} {(B, S, Dn, Dr)}"
    # untouched rows: bit for bit
    np.testing.assert_array_equal(got_n[~written], inputs.to_numpy(cn_cpu)[~written], what)
    np.testing.assert_array_equal(got_r[~written], inputs.to_numpy(cr_cpu)[~written], what)
    if dtype != "f32":
        assert_rounded_close(got_n[written], want_n[written], dtype, what + " norm")
        assert_rounded_close(got_r[written], want_r[written], dtype, what + " rope")
    else:
        # fp32: compare with the unrounded fp64 results of the two pinned operators
        kvs = inputs.to_numpy(kv_cpu).astype(np.float64)
        for t in range(B * S):
            slot = int(s_np[t])
            if not 0 <= slot < ns:
                continue
            b, s_ = divmod(t, S)
            ref_n = oracle.rmsnorm_f64(kvs[b, s_, None, :Dn],
                                       inputs.to_numpy(gamma_cpu).astype(np.float64),
                                       float(np.float32(1e-5)))[0]
            ref_r = oracle.rope_f64(kvs[b, s_, None, None, None, Dn:], sin_cpu.numpy()[s_:s_ + 1],
                                    cos_cpu.numpy()[s_:s_ + 1])[0, 0, 0]
            assert_f32_close(got_n[slot], ref_n, what + " norm")
            assert_f32_close(got_r[slot], ref_r, what + " rope")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(2, 300, 512, 64), (1, 7, 512, 64), (3, 17, 128, 32),
                                   (2, 9, 33, 6), (1, 5, 1000, 128), (2, 4, 8, 2)])
def test_shapes(shape, dtype):
    run_case(*shape, dtype, seed=sum(shape))


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_variant(dtype):
    es = ES[dtype]
    # (norm access bytes, norm accesses per lane, rope access bytes per half and lane)
    variants = [(16, nvn, rb) for nvn in (1, 2, 4, 8) for rb in (4, 8, 16) if rb >= 2 * es]
    variants += [(es, nvn, es) for nvn in (1, 2, 4, 8, 16)]
    for vb, nvn, rb in variants:
        e, re = vb // es, rb // es
        Dn = max(e, (32 * nvn - 1) * e)              # one access short: a ragged last lane
        for lanes in (6, 32):                        # a few rope lanes, and a full warp
            Dr = 2 * re * lanes
            plan = camp.Plan(kernel=camp.KERNEL_KV_CACHE, vec_bytes=vb, per_thread=nvn,
                             group=rb)
            run_case(2, 6, Dn, Dr, dtype, seed=vb * nvn + rb + lanes, plan=plan)


def test_many_tokens_uses_the_table_row_of_each_position():
    # 3 x 1500 tokens: the table row is t mod S for every token (multiply-shift division)
    run_case(3, 1500, 64, 64, "bf16", seed=11, pad=True)


def test_no_padding_full_cache():
    run_case(1, 256, 512, 64, "bf16", seed=3, num_slots=256, pad=False)


def test_mla_shaped_large():
    run_case(1, 4096, 512, 64, "bf16", seed=5)
