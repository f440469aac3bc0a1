"""Pins the tcgen05 encodings the MLA kernel relies on (shared-memory
descriptors, instruction descriptor, A operand in tensor memory) with tiny
single-CTA MMAs whose results are checked against torch matmul."""

import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = str(tmp_path_factory.mktemp("probe") / "libumma_probe.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "--cudart", "shared",
                    "-I" + os.path.join(ROOT, "paged_kv_decode_20_gb300", "csrc"),
                    os.path.join(HERE, "gpu_probes", "umma_probe.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.umma_probe.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.umma_probe.restype = ctypes.c_int
    return lib


def _run(lib, mode, A, B, n, lbo=16, sbo=1024):
    D = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.umma_probe(mode, A.data_ptr(), B.data_ptr(), D.data_ptr(), lbo, sbo, st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    return D


def _rand(*shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)


def test_kmajor_ss(probe):
    A, B = _rand(128, 64, seed=1), _rand(64, 64, seed=2)
    D = _run(probe, 0, A, B, 64)
    torch.testing.assert_close(D, A.float() @ B.float().T, rtol=1e-4, atol=1e-3)


def test_b_mn_major_leading_offset_is_the_column_chunk_stride(probe):
    A, V = _rand(128, 64, seed=3), _rand(64, 256, seed=4)
    D = _run(probe, 1, A, V, 256, lbo=8192, sbo=1024)
    torch.testing.assert_close(D, A.float() @ V.float(), rtol=1e-4, atol=1e-3)


def test_a_from_tensor_memory(probe):
    A, B = _rand(128, 64, seed=5), _rand(64, 64, seed=6)
    D = _run(probe, 2, A, B, 64)
    torch.testing.assert_close(D, A.float() @ B.float().T, rtol=1e-4, atol=1e-3)


def _rand_e4m3(*shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(*shape, generator=g, device="cuda") * 4).to(torch.float8_e4m3fn)


def test_e4m3_kmajor_ss(probe):
    """kind::f8f6f4 with E4M3 A and B, K-major, 128-byte swizzle: four K = 32 steps."""
    A, B = _rand_e4m3(128, 128, seed=7), _rand_e4m3(64, 128, seed=8)
    D = _run(probe, 3, A, B, 64)
    torch.testing.assert_close(D, A.float() @ B.float().T, rtol=1e-4, atol=1e-3)


def test_e4m3_a_from_tensor_memory(probe):
    A, B = _rand_e4m3(128, 128, seed=9), _rand_e4m3(64, 128, seed=10)
    D = _run(probe, 4, A, B, 64)
    torch.testing.assert_close(D, A.float() @ B.float().T, rtol=1e-4, atol=1e-3)


def test_e4m3_kmajor_64_byte_swizzle(probe):
    """64-byte rows (the rope part of an E4M3 latent row) with the 64-byte swizzle."""
    A, B = _rand_e4m3(128, 64, seed=11), _rand_e4m3(64, 64, seed=12)
    D = _run(probe, 5, A, B, 64)
    torch.testing.assert_close(D, A.float() @ B.float().T, rtol=1e-4, atol=1e-3)


def test_f16_b_mn_major(probe):
    g = torch.Generator(device="cuda").manual_seed(13)
    A = torch.rand(128, 64, generator=g, device="cuda").to(torch.float16)
    V = torch.randn(64, 256, generator=g, device="cuda").to(torch.float16)
    D = _run(probe, 6, A, V, 256, lbo=8192, sbo=1024)
    torch.testing.assert_close(D, A.float() @ V.float(), rtol=1e-4, atol=1e-3)
