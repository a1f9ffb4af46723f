"""Seeded synthetic inputs for RMSNorm and RoPE.

This module holds no arithmetic of either operator. It draws the inputs that the CUDA
path and the CPU oracle both consume, so that the two are compared on identical data:

* RMSNorm: ``x[rows, cols] ~ N(0, 1)``, ``w[cols] ~ N(1, 0.1)``; in the stress recipe
  1% of the rows (chosen by a seeded permutation) are scaled by 1e3 and another,
  disjoint 1% by 1e-4. Values are drawn in fp32 and rounded once to the storage type
  (bf16 and fp16 rounding is torch's, round to nearest even; in fp16 the 1e-4 rows are
  partly subnormal).
* RoPE: ``x[B, S, H, D] ~ N(0, 1)`` rounded to the storage type, and fp32 tables
  ``sin, cos [S, D/2]`` at ``angle = s * theta^(-2i/D)``, ``i = 0 .. D/2-1``, computed in
  fp64 and rounded once to fp32 (Llama-3.2-1B uses theta = 500000).

* LayerNorm: ``x[r, :] = o_r + s_r * N(0, 1)`` with a per-row scale ``s_r`` drawn from
  {1e-2, 1, 10} and an offset ratio ``o_r / s_r`` from {0, +-3, +-100} (bf16, fp16) or
  {0, +-3, +-1e3} (fp32), so some rows have |mean| >> spread; ``gamma ~ N(1, 0.1)``,
  ``beta ~ N(0, 1)`` (beta and gamma * xhat then cancel somewhere in every long row).

Sub-seeds: x uses ``seed*16 + 0``, w ``seed*16 + 1``, the stress-row permutation
``seed*16 + 2``, the RoPE input ``seed*16 + 3``, and the LayerNorm beta ``seed*16 + 4``
and row scales and offsets ``seed*16 + 5``. ``device`` selects where the numbers
are drawn (torch's CPU and CUDA generators give different streams for one seed; the
recipe is the distribution, and every comparison uses one draw for both sides).
"""

from __future__ import annotations

import numpy as np
import torch

STORAGE = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _gen(seed: int, k: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + k)
    return g


def rmsnorm_inputs(rows: int, cols: int, dtype: str = "bf16", seed: int = 0,
                   stress: bool = False, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Return ``(x[rows, cols], w[cols])`` of storage type ``dtype`` on ``device``."""
    st = STORAGE[dtype]
    x = torch.randn(rows, cols, generator=_gen(seed, 0, device), dtype=torch.float32,
                    device=device)
    w = torch.randn(cols, generator=_gen(seed, 1, device), dtype=torch.float32,
                    device=device)
    w = w.mul_(0.1).add_(1.0)
    if stress and rows > 0:
        n1 = rows // 100
        perm = torch.randperm(rows, generator=_gen(seed, 2, "cpu")).to(device)
        if n1 > 0:
            x[perm[:n1]] *= 1e3
            x[perm[n1:2 * n1]] *= 1e-4
    return x.to(st), w.to(st)


def layernorm_inputs(rows: int, cols: int, dtype: str = "bf16", seed: int = 0,
                     device="cpu") -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Return ``(x[rows, cols], gamma[cols], beta[cols])`` of storage type ``dtype``."""
    st = STORAGE[dtype]
    x = torch.randn(rows, cols, generator=_gen(seed, 0, device), dtype=torch.float32,
                    device=device)
    g = torch.randn(cols, generator=_gen(seed, 1, device), dtype=torch.float32, device=device)
    g = g.mul_(0.1).add_(1.0)
    b = torch.randn(cols, generator=_gen(seed, 4, device), dtype=torch.float32, device=device)
    pick = torch.randint(0, 1 << 30, (rows, 2), generator=_gen(seed, 5, "cpu"))
    scales = torch.tensor([1e-2, 1.0, 10.0])
    ratios = torch.tensor([0.0, 3.0, -3.0, 1e3, -1e3] if dtype == "f32"
                          else [0.0, 3.0, -3.0, 100.0, -100.0])
    s_r = scales[pick[:, 0] % len(scales)]
    o_r = ratios[pick[:, 1] % len(ratios)] * s_r
    x = x * s_r.to(device)[:, None] + o_r.to(device)[:, None]
    return x.to(st), g.to(st), b.to(st)


def rope_tables(S: int, D: int, theta: float = 500000.0) -> tuple[np.ndarray, np.ndarray]:
    """fp32 ``(sin, cos)`` tables ``[S, D/2]``: angle = s * theta^(-2i/D), drawn in fp64."""
    half = D // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / D)
    angle = np.arange(S, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.sin(angle).astype(np.float32), np.cos(angle).astype(np.float32)


def rope_inputs(B: int, S: int, H: int, D: int, dtype: str = "bf16", seed: int = 0,
                theta: float = 500000.0, device="cpu"
                ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Return ``(x[B, S, H, D], sin[S, D/2], cos[S, D/2])``; x of ``dtype``, tables fp32."""
    st = STORAGE[dtype]
    x = torch.randn(B, S, H, D, generator=_gen(seed, 3, device), dtype=torch.float32,
                    device=device).to(st)
    sin_t, cos_t = rope_tables(S, D, theta)
    return x, torch.from_numpy(sin_t).to(device), torch.from_numpy(cos_t).to(device)


def p3_style_rmsnorm_inputs(rows: int, cols: int, dtype: str = "bf16"
                            ) -> tuple[torch.Tensor, torch.Tensor]:
    """Deterministic RMSNorm case in the style of the xserv unit tests:
    ``x_i = ((i mod 17) - 8) * 0.1`` over the flattened matrix, ``w_j = 0.5 + (j mod 3) * 0.2``."""
    i = torch.arange(rows * cols, dtype=torch.float32)
    x = (((i % 17) - 8.0) * 0.1).reshape(rows, cols)
    w = 0.5 + (torch.arange(cols, dtype=torch.float32) % 3) * 0.2
    return x.to(STORAGE[dtype]), w.to(STORAGE[dtype])


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """CPU copy as numpy: bf16 as ``uint16`` bit patterns, fp16 as ``float16``, fp32 as
    ``float32``."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def from_numpy(a: np.ndarray) -> torch.Tensor:
    """Inverse of :func:`to_numpy` (``uint16`` is read as bf16 bit patterns, ``float16`` as
    fp16)."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))
