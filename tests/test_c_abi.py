"""The C ABI from C: `tests/c_consumer.c`, a plain C11 program with CUDA-runtime buffers and
a stream of its own, built against `include/camp.h` and `libcamp.so`.

Without a GPU: the header compiles as strict C99 and C11, and the consumer compiles and
links. On the GPU: the consumer runs RMSNorm (fp32) and RoPE (bf16) through the ABI, checks
argument errors from C, and its outputs are compared with the oracle (fp32 within
1e-6 + 2e-6 |ref| of the fp64 result, bf16 within 1 ulp of the result rounded once).
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from block_memory_bound_gb300 import build, camp, inputs
from parity import assert_bf16_close, assert_f32_close

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "c_consumer.c")


def _cuda_dirs():
    home = os.environ.get("CUDA_HOME") or os.path.dirname(os.path.dirname(build.nvcc()))
    libs = [os.path.join(home, "lib64")] + glob.glob(os.path.join(home, "targets", "*", "lib"))
    lib = next((d for d in libs if glob.glob(os.path.join(d, "libcudart.so*"))), None)
    return os.path.join(home, "include"), lib


def _cc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    return cc


def _build_consumer(out: str) -> str:
    inc, lib = _cuda_dirs()
    if lib is None:
        pytest.skip("no libcudart.so next to the CUDA toolkit")
    camp_lib = build.build()
    cmd = [_cc(), "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", build.INCLUDE,
           "-I", inc, SOURCE, "-o", out, "-L", os.path.dirname(camp_lib), "-lcamp",
           "-L", lib, "-lcudart", f"-Wl,-rpath,{os.path.dirname(camp_lib)}:{lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


@pytest.mark.parametrize("std", ["c99", "c11"])
def test_header_is_strict_c(tmp_path, std):
    src = tmp_path / "h.c"
    src.write_text('#include "camp.h"\nint main(void) { return (int)CAMP_SUCCESS; }\n')
    r = subprocess.run([_cc(), f"-std={std}", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", build.INCLUDE, "-fsyntax-only", str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_consumer_compiles_and_links(tmp_path):
    exe = _build_consumer(str(tmp_path / "c_consumer"))
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_consumer_runs_through_the_c_abi(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    camp.load()
    exe = _build_consumer(str(tmp_path / "c_consumer"))
    rows, cols, B, S, H, D = 37, 3000, 2, 33, 8, 64
    x, w = inputs.rmsnorm_inputs(rows, cols, "f32", seed=11)
    q, sn, cs = inputs.rope_inputs(B, S, H, D, "bf16", seed=12)
    xs, ws = inputs.to_numpy(x), inputs.to_numpy(w)
    qs, sns, css = inputs.to_numpy(q), sn.numpy(), cs.numpy()
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(src, "wb") as f:
        f.write(np.array([rows, cols, B, S, H, D], dtype=np.int64).tobytes())
        for a in (xs, ws, qs, sns, css):
            f.write(np.ascontiguousarray(a).tobytes())
    r = subprocess.run([exe, str(src), str(dst)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    raw = open(dst, "rb").read()
    ny = rows * cols * 4
    assert len(raw) == ny + q.numel() * 2
    y = np.frombuffer(raw[:ny], dtype=np.float32).reshape(rows, cols)
    yq = np.frombuffer(raw[ny:], dtype=np.uint16).reshape(B, S, H, D)
    ref = oracle.rmsnorm_f64(xs.astype(np.float64), ws.astype(np.float64),
                             float(np.float32(1e-5)))
    assert_f32_close(y, ref, "rmsnorm fp32 from C")
    assert_bf16_close(yq, oracle.rope(qs, sns, css, "bf16"), "rope bf16 from C")
