"""tcgen05 operand conventions of the fused pass's column-block scores: a K-major B
operand in the no-swizzle core-matrix layout (the score blocks the intra MMA reads),
and the N = 16 score product whose 64 query rows sit in rows 64-127 of an M = 128
operand and are read back from tensor-memory lanes 64-127. Each is one MMA
pipeline compared with torch on the same bf16 inputs."""
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
    so = os.path.join(OUT, "libumma_probe2.so")
    src = os.path.join(HERE, "csrc", "umma_probe2.cu")
    subprocess.check_call([gbuild.nvcc(), *gbuild.ARCH, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                           "--cudart", "static", "-I", gbuild.CSRC, "-o", so, src])
    lib = ctypes.CDLL(so)
    lib.umma_probe2.restype = ctypes.c_int
    lib.umma_probe2.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p]
    return lib


def _rand(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16).cuda()


def test_no_swizzle_k_major_blocks(probe):
    V, P = _rand(64, 128, seed=11), _rand(64, 64, seed=12)
    ref = V.float().T @ P.float().T
    D = torch.full(ref.shape, float("nan"), device="cuda")
    assert probe.umma_probe2(3, 0, 0, V.data_ptr(), P.data_ptr(), D.data_ptr()) == 0
    err = (D - ref).abs().max().item() / ref.abs().max().item()
    if not err < 1e-5:
        D2 = torch.full(ref.shape, float("nan"), device="cuda")
        probe.umma_probe2(3, 0, 1, V.data_ptr(), P.data_ptr(), D2.data_ptr())
        err2 = (D2 - ref).abs().max().item() / ref.abs().max().item()
        pytest.fail(f"no-swizzle blocks: err {err:.3e}; with LBO/SBO swapped: {err2:.3e}")


@pytest.mark.parametrize("c", [0, 1, 2, 3])
def test_column_block_scores_in_upper_lanes(probe, c):
    Q, K = _rand(64, 256, seed=13), _rand(64, 256, seed=14)
    ref = Q.float() @ K.float()[16 * c:16 * c + 16].T
    D = torch.full(ref.shape, float("nan"), device="cuda")
    assert probe.umma_probe2(4, c, 0, Q.data_ptr(), K.data_ptr(), D.data_ptr()) == 0
    err = (D - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, f"column block {c}: max rel err {err:.3e}"
