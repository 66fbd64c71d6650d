"""GPU parity of the phase-1 projection GEMM (la_gemm_bf16: C = A W^T on the tensor cores)
against the fp64 oracle, over shapes with tails in M, N and K, a single row, exact tiles,
strided operands, and shapes with several times more 128 x 256 tiles than the GPU has SMs, so
that every persistent block walks several tiles (both TMEM accumulators, barrier phases carried
from tile to tile).

Bar (derived from the arithmetic): the output is rounded to bf16 once (relative error 2^-9) after
an fp32 accumulation over K products (error at most K 2^-24 sum_k |a_mk w_nk|), so
|c - c_ref| <= 2^-8 |c_ref| + K 2^-24 sum_k |a_mk w_nk|.
"""
import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
from tests.helpers import f64
import oracle

pytestmark = pytest.mark.gpu


def check(a, w, c):
    ref = oracle.linear(f64(a), f64(w))
    mag = np.abs(f64(a)) @ np.abs(f64(w)).T
    K = a.shape[1]
    err = np.abs(f64(c) - ref)
    bound = 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -24 * mag
    assert np.all(err <= bound), float((err - bound).max())
    return float(err.max())


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (1, 8, 8), (128, 256, 64), (257, 256, 1000),
                                   (129, 7 * 256 + 8, 136), (2048, 1024, 2048)])
def test_gemm_matches_oracle(cuda, M, N, K):
    g = torch.Generator("cpu")
    g.manual_seed(M + N + K)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    c = torch.full((M, N), 9.0, dtype=torch.bfloat16, device=cuda)
    la.gemm_bf16(a.to(cuda), w.to(cuda), c)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    e = check(a, w, c.cpu())
    print(f"\n[parity] gemm {M}x{N}x{K}: max|c-c_ref| = {e:.3e}")


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 2048), (4000, 4104, 520)])
def test_gemm_multi_tile_per_block_matches_oracle(cuda, M, N, K):
    """512 (and 32 x 17 = 544, with tails in M, N and K) output tiles on the GPU's SMs: every block runs its
    tile loop several times. The oracle is evaluated on a sample of rows from every row band
    (the first and last row of each 128-row band and one inside it) against all columns."""
    tiles = ((M + 127) // 128) * ((N + 255) // 256)
    assert tiles > 2 * torch.cuda.get_device_properties(cuda).multi_processor_count
    g = torch.Generator("cpu")
    g.manual_seed(M + N + K + 1)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    c = torch.full((M, N), 9.0, dtype=torch.bfloat16, device=cuda)
    la.gemm_bf16(a.to(cuda), w.to(cuda), c)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    rows = sorted({r for m0 in range(0, M, 128) for r in (m0, min(m0 + 77, M - 1),
                                                          min(m0 + 127, M - 1))})
    e = check(a[rows], w, c.cpu()[rows])
    print(f"\n[parity] gemm {M}x{N}x{K} ({tiles} tiles): max|c-c_ref| = {e:.3e} "
          f"over {len(rows)} rows")


def test_gemm_strided_operands_and_guard(cuda):
    g = torch.Generator("cpu")
    g.manual_seed(7)
    M, N, K = 200, 300, 120
    a_full = torch.randn(M, K + 24, generator=g).to(torch.bfloat16).to(cuda)
    w_full = torch.randn(N, K + 8, generator=g).to(torch.bfloat16).to(cuda)
    c_full = torch.full((M + 3, N + 20), 4.0, dtype=torch.bfloat16, device=cuda)
    a, w, c = a_full[:, :K], w_full[:, :K], c_full[:M, :N]
    la.gemm_bf16(a, w, c)
    torch.cuda.synchronize()
    check(a.cpu(), w.cpu(), c.cpu())
    assert torch.all(c_full[M:].cpu() == 4.0) and torch.all(c_full[:, N:].cpu() == 4.0)


def test_gemm_twice_same_bits(cuda):
    g = torch.Generator("cpu")
    g.manual_seed(8)
    a = torch.randn(640, 512, generator=g).to(torch.bfloat16).to(cuda)
    w = torch.randn(768, 512, generator=g).to(torch.bfloat16).to(cuda)
    c1, c2 = la.gemm_bf16(a, w), la.gemm_bf16(a, w)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
