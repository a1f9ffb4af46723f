"""The byte/FLOP ledger against the numbers the pages print (tests/golden/ledger_pages.txt)."""

from __future__ import annotations

import os

import pytest

from block_memory_bound_gb300 import ledger

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ledger_pages.txt")


def _golden() -> dict[str, str]:
    out = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            fields = [f.strip() for f in line.split("|")]
            out[fields[0]] = fields[3]
    return out


def test_rope_ledger_matches_tutorial_e13():
    g = _golden()
    flops = ledger.rope_flops(1, 4096, 32, 128)
    nbytes = ledger.rope_bytes(1, 4096, 32, 128, "fp16", tables=False)
    assert round(flops / 1e6, 1) == float(g["rope_e13_flops"])
    assert round(nbytes / 1e6, 2) == float(g["rope_e13_bytes"])
    assert round(flops / nbytes, 2) == float(g["rope_e13_ai"])
    t = ledger.time_lower_bound_s(nbytes, flops, 4502e9, 729e12)
    assert round(t * 1e6, 1) == float(g["rope_e13_tlb"])


@pytest.mark.parametrize("key", ["rms_ninetoothed", "rms_tilelang", "rms_torch"])
def test_rmsnorm_effective_bandwidth_matches_gollamago_table(key):
    ms, gbs = (float(v) for v in _golden()[key].split(","))
    nbytes = ledger.rmsnorm_bytes(4096, 2048, "bf16", weight=False)
    assert round(nbytes / (ms * 1e-3) / 1e9) == pytest.approx(gbs, abs=1)


def test_layernorm_ledger_matches_tutorial_example_2():
    g = _golden()
    fused = ledger.layernorm_bytes(8192, 4096, "fp16", affine=False)
    split = ledger.layernorm_bytes(8192, 4096, "fp16", affine=False, passes=3)
    assert round(fused / 1e6, 1) == float(g["ln_ex2_fused_bytes"])
    assert round(split / 1e6, 1) == float(g["ln_ex2_unfused_bytes"])
    assert round(ledger.layernorm_flops(8192, 4096) / 1e9, 3) == float(g["ln_ex2_flops"])
    # with gamma and beta read once each, as reported by the benchmark
    assert ledger.layernorm_bytes(8192, 4096, "fp16") == fused + 2 * 4096 * 2


def test_benchmark_step_bytes():
    # RMSNorm bf16 [4096, 2048] + RoPE Q [1,4096,32,64] + RoPE K [1,4096,8,64], with the
    # weight and the fp32 tables counted once per launch.
    assert ledger.rmsnorm_bytes(4096, 2048) == 33_558_528
    assert ledger.rope_bytes(1, 4096, 32, 64) == 34_603_008
    assert ledger.rope_bytes(1, 4096, 8, 64) == 9_437_184
    # fused Q + K: the shared tables counted once
    assert ledger.rope_qk_bytes(1, 4096, 32, 8, 64) == 42_991_616
    assert ledger.rmsnorm_bytes(16384, 8192) == 536_887_296
    assert ledger.rmsnorm_bytes(64, 2048, "f32") == 1_056_768


def test_kv_cat_repeat_bytes():
    # Llama-3.2-1B keys, 4096 positions (3584 cached + 512 new), 8 heads of 64 repeated 4
    # times: 4096*8*64*2 bytes read, four times that written, 512 table rows of 32 sin + cos.
    rows = 4096 * 8 * 64 * 2
    assert ledger.kv_cat_repeat_bytes(1, 3584, 512, 8, 64, 4) == 5 * rows + 2 * 512 * 32 * 4
    assert ledger.kv_cat_repeat_bytes(1, 3584, 512, 8, 64, 4, tables=False) == 5 * rows
    assert ledger.kv_cat_repeat_bytes(2, 5, 0, 2, 8, 3, "f32") == 2 * 5 * 2 * 8 * 4 * 4
