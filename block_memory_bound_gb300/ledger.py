"""Algorithmic bytes and FLOPs per launch (the roofline numerators).

Accounting rules (tilelang tutorial ch. 02, section 2.1): every input is read once and
every output written once; intermediates are not counted; an elementary operation or a
transcendental counts 1 FLOP, a multiply-add 2. The roofline time bound is
max(bytes / bandwidth, flops / peak).

The pages' own RoPE ledger (ch. 02, exercise E13) leaves the precomputed sin/cos
tables out; the gollamago effective-bandwidth figures count only the x read and the y
write of RMSNorm. The numbers reported here include the weight and the tables
(``weight=True``, ``tables=True``): each is read once per launch as well.
"""

from __future__ import annotations

ELEM_BYTES = {"bf16": 2, "f16": 2, "fp16": 2, "f32": 4, "fp32": 4}


def rmsnorm_bytes(rows: int, cols: int, dtype: str = "bf16", weight: bool = True) -> int:
    es = ELEM_BYTES[dtype]
    return 2 * rows * cols * es + (cols * es if weight else 0)


def add_rmsnorm_bytes(rows: int, cols: int, dtype: str = "bf16") -> int:
    """Fused residual add + RMSNorm: x and r read once, h and y written once, w read once."""
    es = ELEM_BYTES[dtype]
    return 4 * rows * cols * es + cols * es


def layernorm_bytes(rows: int, cols: int, dtype: str = "bf16", affine: bool = True,
                    passes: int = 1) -> int:
    """LayerNorm: x read ``passes`` times (1 when fused; the three-pass split of mean,
    variance and normalize + affine reads it 3 times), y written once, gamma and beta read
    once (``affine=True``; the tutorial's example 2 leaves them out)."""
    es = ELEM_BYTES[dtype]
    return (passes + 1) * rows * cols * es + (2 * cols * es if affine else 0)


def layernorm_flops(rows: int, cols: int) -> int:
    # the tutorial's convention for example 2: about 8 FLOP per element
    return 8 * rows * cols


def rmsnorm_flops(rows: int, cols: int) -> int:
    # per element: square-accumulate (2) + two multiplies (2); per row: divide, add, rsqrt
    return 4 * rows * cols + 3 * rows


def rope_bytes(B: int, S: int, H: int, D: int, dtype: str = "bf16", tables: bool = True) -> int:
    es = ELEM_BYTES[dtype]
    return 2 * B * S * H * D * es + (2 * S * (D // 2) * 4 if tables else 0)


def rope_qk_bytes(B: int, S: int, Hq: int, Hk: int, D: int, dtype: str = "bf16") -> int:
    """Q and K rotated in one launch: both tensors read and written once, the shared
    tables read once."""
    es = ELEM_BYTES[dtype]
    return 2 * B * S * (Hq + Hk) * D * es + 2 * S * (D // 2) * 4


def kv_cache_bytes(B: int, S: int, Dn: int, Dr: int, dtype: str = "bf16") -> int:
    """KV RMSNorm + RoPE + cache scatter with every token written: kv read once, both cache
    rows written once, gamma, the tables and the int64 slot array read once."""
    es = ELEM_BYTES[dtype]
    return 2 * B * S * (Dn + Dr) * es + Dn * es + 2 * S * (Dr // 2) * 4 + 8 * B * S


def kv_cat_repeat_bytes(B: int, P: int, S: int, Hk: int, D: int, n_rep: int,
                        dtype: str = "bf16", tables: bool = True) -> int:
    """KV concatenation + head repeat: past and new rows read once, every one of the n_rep
    copies of each row written once, the table rows of the new positions read once."""
    es = ELEM_BYTES[dtype]
    return (B * (P + S) * Hk * D * es * (1 + n_rep)
            + (2 * S * (D // 2) * 4 if tables and S > 0 else 0))


def rope_flops(B: int, S: int, H: int, D: int) -> int:
    # per pair: 4 multiplies + 2 add/sub = 6 FLOP, i.e. 3 FLOP per element
    return 3 * B * S * H * D


def time_lower_bound_s(nbytes: float, flops: float, bw_bytes_per_s: float,
                       peak_flops: float) -> float:
    return max(nbytes / bw_bytes_per_s, flops / peak_flops)
