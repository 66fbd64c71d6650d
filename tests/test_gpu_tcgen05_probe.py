"""GPU unit check of the tcgen05 helpers (descriptors, instruction descriptors, TMEM
load/store, MMA from shared and tensor memory, tf32 and bf16, the latter packed two per TMEM
column when it is the A operand) on exactly representable operands, so the product must match
exactly. Shapes are those the recurrence kernel issues."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tc_probe", "probe.cu")
SRC_MN = os.path.join(HERE, "tc_probe", "probe_mn.cu")
CSRC = os.path.join(os.path.dirname(HERE), "linear_attention_chunked_conv1d_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(cuda):
    out_dir = os.path.join(HERE, "tc_probe", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libprobe.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", CSRC, SRC,
                           SRC_MN, "-o", so])
    lib = ctypes.CDLL(so)
    lib.probe_run.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    lib.probe_mn_run.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    return lib


@pytest.mark.parametrize("mode,N,K", [(0, 64, 128), (0, 128, 128), (0, 256, 64),
                                      (1, 128, 128), (1, 64, 64), (2, 128, 128), (2, 64, 64),
                                      (2, 128, 64), (3, 128, 128), (3, 64, 64), (3, 256, 64)])
def test_tcgen05_mma_exact(probe, cuda, mode, N, K):
    g = torch.Generator("cpu")
    g.manual_seed(mode * 1000 + N + K)
    A = torch.randint(-8, 9, (128, K), generator=g).float() / 8
    B = torch.randint(-8, 9, (N, K), generator=g).float() / 8
    D = torch.full((128, N), float("nan"), device=cuda)
    err = torch.zeros(1, dtype=torch.int32, device=cuda)
    Ad, Bd = A.to(cuda), B.to(cuda)
    rc = probe.probe_run(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), N, K, mode, err.data_ptr())
    assert rc == 0 and int(err.item()) == 0
    ref = (A.double() @ B.double().T).float()
    assert torch.equal(D.cpu(), ref), (D.cpu() - ref).abs().max()


def _mn_run(probe, cuda, mode, N, K, swap):
    g = torch.Generator("cpu")
    g.manual_seed(7 * mode + N + K)
    A = torch.randint(-8, 9, (128, K), generator=g).float() / 8
    B = torch.randint(-8, 9, (N, K), generator=g).float() / 8
    # mode 0/1: B passed transposed ([K][N]); mode 2: A passed transposed ([K][128])
    Ain = A.T.contiguous() if mode == 2 else A
    Bin = B if mode == 2 else B.T.contiguous()
    D = torch.full((128, N), float("nan"), device=cuda)
    err = torch.zeros(1, dtype=torch.int32, device=cuda)
    Ad, Bd = Ain.to(cuda), Bin.to(cuda)
    rc = probe.probe_mn_run(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), N, K, mode, swap,
                            err.data_ptr())
    assert rc == 0 and int(err.item()) == 0
    ref = (A.double() @ B.double().T).float()
    return torch.equal(D.cpu(), ref)


@pytest.mark.parametrize("mode,N,K", [(1, 128, 64), (1, 64, 128), (2, 64, 128), (2, 128, 64),
                                      (4, 128, 64), (4, 64, 128)])
def test_tcgen05_mma_mn_major_bf16(probe, cuda, mode, N, K):
    """bf16 MN-major operand (mode 4: with A in tensor memory): leading byte offset = distance
    between 128-byte atoms along M/N, stride byte offset = distance between 8-row groups along
    K."""
    assert _mn_run(probe, cuda, mode, N, K, swap=0)
