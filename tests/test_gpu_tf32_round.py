"""GPU checks of the integer fp32 -> tf32 rounding used by the tensor-core recurrence (round to
nearest, ties away from zero, on the bit pattern):
- against the hardware conversion (cvt.rna.tf32.f32): every non-NaN fp32 bit pattern must give
  the same bits, for the full rounding and for the operand form with its low 13 bits cleared;
- that the tf32 MMA reads only the top 19 bits of an operand, from shared memory and from tensor
  memory (the operand form leaves the low bits set): D = A.I returns each A element with its
  low 13 bits cleared."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tc_probe", "round_probe.cu")
CSRC = os.path.join(os.path.dirname(HERE), "linear_attention_chunked_conv1d_gb300", "csrc")


def test_tf32_rounding_matches_hardware_conversion(cuda):
    out_dir = os.path.join(HERE, "tc_probe", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libround_probe.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", CSRC, SRC,
                           "-o", so])
    lib = ctypes.CDLL(so)
    lib.round_run.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    count = torch.zeros(1, dtype=torch.int64, device=cuda)
    first = torch.full((1,), -1, dtype=torch.int32, device=cuda)  # 0xFFFFFFFF as unsigned
    assert lib.round_run(count.data_ptr(), first.data_ptr()) == 0
    n, b = int(count.item()), int(first.item()) & 0xFFFFFFFF
    assert n == 0, f"{n} patterns differ, the smallest 0x{b:08x}"


@pytest.fixture(scope="module")
def trunc_lib(cuda):
    out_dir = os.path.join(HERE, "tc_probe", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libtrunc_probe.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", CSRC,
                           os.path.join(HERE, "tc_probe", "trunc_probe.cu"), "-o", so])
    lib = ctypes.CDLL(so)
    lib.trunc_run.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    return lib


@pytest.mark.parametrize("from_tmem", [0, 1])
def test_tf32_mma_reads_top_19_bits(trunc_lib, cuda, from_tmem):
    g = torch.Generator("cpu")
    g.manual_seed(11 + from_tmem)
    for _ in range(4):
        bits = torch.randint(0, 2 ** 31, (128 * 8,), generator=g, dtype=torch.int64)
        sign = torch.randint(0, 2, (128 * 8,), generator=g, dtype=torch.int64) << 31
        expo = torch.randint(64, 191, (128 * 8,), generator=g, dtype=torch.int64) << 23
        pat = sign | expo | (bits & 0x7FFFFF)  # normal, finite values with random low bits
        a = torch.tensor(pat.to(torch.int64).numpy().astype("uint32").view("float32"))
        d = torch.zeros(128 * 8, dtype=torch.float32, device=cuda)
        err = torch.zeros(1, dtype=torch.int32, device=cuda)
        assert trunc_lib.trunc_run(a.to(cuda).data_ptr(), d.data_ptr(), from_tmem, err.data_ptr()) == 0
        assert int(err.item()) == 0
        got = d.cpu().numpy().view("uint32")
        want = (pat & 0xFFFFE000).numpy().astype("uint32")
        assert (got == want).all(), int((got != want).sum())
