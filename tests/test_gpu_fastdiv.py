"""The quantizer's correctly rounded reciprocal and division helpers
(csrc/fastdiv.cuh: one Newton step from rcp.approx, Markstein's FMA division
with a correctly rounded reciprocal) against CUDA's IEEE round-to-nearest
__frcp_rn / __fdiv_rn, bit for bit, over every input the quantizer can give
them: every positive finite fp32 for the reciprocal and for the outer scale
s_g = amax / 2688 (or / 1536), every block-scale quotient bmax / (c s_g)
of a bf16 block max and a bf16 row amax, and the block quotient on 2^32
random fp32 pairs.  The E2M1 codes and E4M3 block
scales are decided on these values, so their bit-exactness rests on this.
The sweep kernels live in a test-only CUDA source built here."""
import ctypes
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cuda", "fastdiv_sweep.cu")


@pytest.fixture(scope="module")
def sweep_lib(tmp_path_factory):
    nvcc = os.environ.get("NVCC", shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc")
    out = str(tmp_path_factory.mktemp("fastdiv") / "libfastdiv_sweep.so")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", SRC, "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    L = ctypes.CDLL(out)
    L.fastdiv_sweep.restype = ctypes.c_int
    u64p = ctypes.POINTER(ctypes.c_ulonglong)
    L.fastdiv_sweep.argtypes = [ctypes.c_int, u64p, u64p, u64p]
    return L


@pytest.mark.parametrize("kind,what", [(0, "rcp_rn vs __frcp_rn, every positive finite fp32"),
                                       (1, "outer_scale(a, 2688) vs __fdiv_rn, every positive finite fp32"),
                                       (2, "outer_scale(a, 1536) vs __fdiv_rn, every positive finite fp32"),
                                       (3, "block-scale quotient vs __fdiv_rn, every bf16 bmax x bf16 amax"),
                                       (4, "block-scale quotient vs __fdiv_rn, 2^32 random fp32 pairs")])
def test_fastdiv_matches_ieee(sweep_lib, kind, what):
    bad, first, count = ctypes.c_ulonglong(), ctypes.c_ulonglong(), ctypes.c_ulonglong()
    rc = sweep_lib.fastdiv_sweep(kind, ctypes.byref(bad), ctypes.byref(first), ctypes.byref(count))
    assert rc == 0, f"CUDA error {rc}"
    assert count.value > 2_000_000_000
    assert bad.value == 0, f"{what}: {bad.value} of {count.value} differ, first at index {first.value:#x}"
