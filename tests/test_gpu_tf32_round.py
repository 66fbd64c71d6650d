"""GPU check of the integer fp32 -> tf32 rounding used by the tensor-core recurrence (round to
nearest, ties away from zero, on the bit pattern) against the hardware conversion
(cvt.rna.tf32.f32): every non-NaN fp32 bit pattern must give the same bits."""
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
