"""The tcgen05 building blocks (shared-memory descriptors in both major-nesses,
the bf16 instruction descriptor, TMEM loads) against a plain fp32 matmul.

The probe is compiled from tests/probes/tc05_probe.cu against the library's own
header, so it exercises exactly the wrappers the kernels use."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "hybrid_linear_attention_kda_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = tmp_path_factory.mktemp("probe") / "libprobe.so"
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", CSRC,
                    os.path.join(ROOT, "tests", "probes", "tc05_probe.cu"), "-o", str(out)],
                   check=True)
    lib = ctypes.CDLL(str(out))
    lib.tc05_probe.restype = ctypes.c_int
    lib.tc05_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    lib.wait_probe.restype = ctypes.c_int
    lib.wait_probe.argtypes = [ctypes.c_longlong, ctypes.c_void_p]
    return lib


CASES = [(16, 64, 0, 0), (64, 128, 0, 0), (192, 128, 0, 0), (256, 128, 0, 0), (128, 64, 0, 0),
         (64, 128, 1, 0), (192, 128, 1, 0), (64, 64, 0, 1), (192, 128, 0, 1), (64, 128, 1, 1),
         (128, 128, 1, 1)]


@pytest.mark.parametrize("N,K,a_mn,b_mn", CASES)
def test_tcgen05_mma_layouts(probe, cuda_device, N, K, a_mn, b_mn):
    g = torch.Generator().manual_seed(N * 1000 + K * 10 + 2 * a_mn + b_mn)
    A = torch.randn((128, K), generator=g).to(torch.bfloat16)
    B = torch.randn((N, K), generator=g).to(torch.bfloat16)
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    D = torch.full((128, N), float("nan"), device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    rc = probe.tc05_probe(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), N, K, a_mn, b_mn, err.data_ptr())
    assert rc == 0
    assert int(err.item()) == 0
    ref = A.double() @ B.double().T
    assert torch.allclose(D.cpu().double(), ref, rtol=1e-4, atol=1e-3), \
        float((D.cpu().double() - ref).abs().max())


def test_bounded_wait_gives_up_and_the_context_stays_usable(probe, cuda_device):
    """The kernels' mbarrier waits are bounded: a wait on a barrier that nothing
    arrives at returns false after its limit (1e6 cycles here, about half a
    millisecond) instead of hanging, and the GPU keeps working afterwards."""
    out = torch.zeros(2, dtype=torch.int64, device=cuda_device)
    assert probe.wait_probe(1_000_000, out.data_ptr()) == 0
    ok, cycles = (int(x) for x in out.cpu())
    assert ok == 0
    assert 1_000_000 <= cycles < 50_000_000
    x = torch.arange(1024, device=cuda_device, dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2
