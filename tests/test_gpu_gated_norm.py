"""GPU parity of the gated RMSNorm epilogue (y = o / sqrt(mean(o^2) + eps) * w * SiLU(z) per
(token, v-head) row): the separate kernel (la_gated_rmsnorm) against the fp64 oracle on the same
o, and the fused output store of la_prefill_front bit for bit against la_prefill_front without z
followed by la_gated_rmsnorm. Together with the recurrence parity tests this pins the whole
chain: o against the oracle within its bar, then the norm on that o within one bf16 ulp.
"""
import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
from tests.helpers import bf16_ulp_diff, f64
import oracle

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def gen(seed):
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    return g


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dv", [64, 128])
def test_gated_rmsnorm_kernel_matches_oracle(cuda, dtype, dv):
    g = gen(dv + (dtype == "bf16"))
    t, Hv = 77, 5
    o = (torch.randn(t, Hv, dv, generator=g) * 0.1).to(DT[dtype])
    z = (torch.randn(t, Hv, dv, generator=g) * 2.0).to(DT[dtype])
    w = (1.0 + 0.3 * torch.randn(dv, generator=g)).to(DT[dtype])
    o[3, 1] = 0  # a zero row: y = 0 (eps keeps it finite)
    y = torch.full_like(o, 9.0).to(cuda)
    la.gated_rmsnorm(o.to(cuda), z.to(cuda), w.to(cuda), y, eps=1e-6)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(f64(o), f64(z), f64(w), 1e-6)
    got = y.cpu()
    if dtype == "bf16":
        assert bf16_ulp_diff(got, ref) <= 1
    else:
        err = np.abs(f64(got) - ref)
        assert np.all(err <= 2e-5 * (1.0 + np.abs(ref))), float(err.max())
    assert torch.all(got[3, 1] == 0)


def test_gated_rmsnorm_in_place(cuda):
    g = gen(5)
    o = (torch.randn(40, 3, 128, generator=g) * 0.2).to(torch.bfloat16).to(cuda)
    z = torch.randn(40, 3, 128, generator=g).to(torch.bfloat16).to(cuda)
    w = torch.ones(128, dtype=torch.bfloat16, device=cuda)
    y = la.gated_rmsnorm(o, z, w, torch.empty_like(o))
    o2 = o.clone()
    la.gated_rmsnorm(o2, z, w)  # in place
    torch.cuda.synchronize()
    assert torch.equal(y, o2)


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("lengths", [[200], [1, 0, 70, 129, 64]])
def test_fused_gated_store_equals_separate_norm(cuda, kda, lengths):
    g = gen(11 + kda + len(lengths))
    Hk, Hv, D, K = 1, 2, 128, 4
    T, B = sum(lengths), len(lengths)
    cd = 2 * Hk * D + Hv * D
    bf = torch.bfloat16
    x = torch.randn(T, cd, generator=g).to(bf).to(cuda)
    w = (torch.randn(cd, K, generator=g) * 0.25).to(bf).to(cuda)
    st0 = torch.randn(B, K - 1, cd, generator=g).to(bf)
    h0 = torch.randn(B, Hv, D, D, generator=g) * 0.02
    gate = -torch.nn.functional.softplus(torch.randn(*((T, Hv, D) if kda else (T, Hv)),
                                                     generator=g)).to(cuda)
    beta = torch.sigmoid(torch.randn(T, Hv, generator=g)).to(cuda)
    z = (torch.randn(T, Hv, D, generator=g) * 2.0).to(bf).to(cuda)
    nw = (1.0 + 0.3 * torch.randn(D, generator=g)).to(bf).to(cuda)
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32, device=cuda)
    ws = torch.empty(la.prefill_workspace_bytes(B, T, Hk, Hv, D, D, bf), dtype=torch.uint8,
                     device=cuda)

    def run(with_z):
        st, h = st0.clone().to(cuda), h0.clone().to(cuda)
        out = torch.full((T, Hv, D), 3.0, dtype=bf, device=cuda)
        la.prefill_front(la.pointer_array([st[s] for s in range(B)]),
                         la.pointer_array([h[s] for s in range(B)]), x, w, gate, beta, out, cu,
                         Hk=Hk, Hv=Hv, dk=D, dv=D, kda=kda, max_seqlen=max(lengths),
                         z=z if with_z else None, norm_w=nw if with_z else None, norm_eps=1e-6,
                         workspace=ws)
        return out, h, st

    o_plain, h1, s1 = run(False)
    y_fused, h2, s2 = run(True)
    y_sep = la.gated_rmsnorm(o_plain, z, nw, torch.empty_like(o_plain), eps=1e-6)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    assert torch.equal(y_fused, y_sep)
    assert torch.equal(h1, h2) and torch.equal(s1, s2)  # the epilogue changes nothing else
    ref = oracle.gated_rmsnorm(f64(o_plain.cpu()), f64(z.cpu()), f64(nw.cpu()), 1e-6)
    assert bf16_ulp_diff(y_fused.cpu(), ref) <= 1
