"""tcgen05 operand-convention probe: the three products the chunk kernel
issues (MN-major x MN-major, MN-major x K-major, TMEM x K-major) computed by
one MMA pipeline and compared with torch on the same bf16 inputs."""
import ctypes
import os
import subprocess

import pytest
import torch

from chunkwise_gated_linear_gla_gb300 import build as gbuild

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "_build")


@pytest.fixture(scope="module")
def probe():
    os.makedirs(OUT, exist_ok=True)
    so = os.path.join(OUT, "libumma_probe.so")
    src = os.path.join(HERE, "csrc", "umma_probe.cu")
    subprocess.check_call([gbuild.nvcc(), *gbuild.ARCH, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                           "--cudart", "static", "-I", gbuild.CSRC, "-o", so, src])
    lib = ctypes.CDLL(so)
    lib.umma_probe.restype = ctypes.c_int
    lib.umma_probe.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return lib


def _rand(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_umma_conventions(probe, mode):
    if mode == 0:
        A, B = _rand(64, 128, seed=1), _rand(64, 256, seed=2)
        ref = A.float().T @ B.float()
    elif mode == 1:
        A, B = _rand(64, 128, seed=3), _rand(64, 64, seed=4)
        ref = A.float().T @ B.float().T
    else:
        A, B = _rand(128, 256, seed=5), _rand(64, 256, seed=6)
        ref = A.float() @ B.float().T
    D = torch.full(ref.shape, float("nan"), device="cuda")
    rc = probe.umma_probe(mode, 0, A.data_ptr(), B.data_ptr(), D.data_ptr())
    assert rc == 0, f"probe status {rc}"
    err = (D - ref).abs().max().item() / ref.abs().max().item()
    if not err < 1e-5 and mode != 2:
        D2 = torch.full(ref.shape, float("nan"), device="cuda")
        probe.umma_probe(mode, 1, A.data_ptr(), B.data_ptr(), D2.data_ptr())
        err2 = (D2 - ref).abs().max().item() / ref.abs().max().item()
        pytest.fail(f"mode {mode}: err {err:.3e}; with LBO/SBO swapped: {err2:.3e}")
    assert err < 1e-5, f"mode {mode}: max rel err {err:.3e}"
