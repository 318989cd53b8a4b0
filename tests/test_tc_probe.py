"""GPU probes of the tcgen05 building blocks (test-only CUDA library): one MMA
tile per operand layout against torch matmul of the same bf16 values."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from paged_mla_speculative_tree_gb300 import build as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tc_probe", "tc_probe.cu")
LIB = os.path.join(HERE, "tc_probe", "libtc_probe.so")


@pytest.fixture(scope="module")
def probe():
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(SRC), os.path.getmtime(
            os.path.join(B.CSRC, "tc_ptx.cuh"))):
        subprocess.check_call([B.nvcc(), *B.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                               "-I", B.CSRC, "-I", B.INCLUDE, SRC, "-o", LIB])
    lib = ctypes.CDLL(LIB)
    lib.tc_probe_run.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 5
    lib.tc_probe_run.restype = ctypes.c_int
    return lib


CASES = {  # variant: (N, K)
    0: (64, 64), 1: (64, 64), 2: (256, 32), 3: (64, 32), 4: (64, 96), 5: (256, 32),
}


def _run(lib, variant):
    N, K = CASES[variant]
    g = torch.Generator().manual_seed(variant)
    A = torch.randn((128, K), generator=g).bfloat16()
    Bm = torch.randn((N, K), generator=g).bfloat16()
    dA, dB = A.cuda(), Bm.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_probe_run(variant, N, K, dA.data_ptr(), dB.data_ptr(), D.data_ptr(), st.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    ref = (A.double() @ Bm.double().T).numpy()
    return D.cpu().double().numpy(), ref


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_probe_layout(probe, variant):
    got, ref = _run(probe, variant)
    err = np.abs(got - ref).max()
    assert err < 1e-3 * max(1.0, np.abs(ref).max()), f"variant {variant}: max err {err}"


def test_probe_mn_major_offsets_identified(probe):
    """Records which LBO/SBO assignment of the MN-major descriptor is right
    (variant 2 is the one the kernel uses; 5 swaps the two offsets)."""
    g2, ref = _run(probe, 2)
    g5, _ = _run(probe, 5)
    ok2 = np.abs(g2 - ref).max() < 1e-3 * np.abs(ref).max()
    ok5 = np.abs(g5 - ref).max() < 1e-3 * np.abs(ref).max()
    print(f"MN-major: lbo=MN-atom stride ok={ok2}; swapped ok={ok5}")
    assert ok2
