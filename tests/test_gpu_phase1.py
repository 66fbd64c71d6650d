"""GPU parity of phase 1 (norm, projections, gates) and of a whole layer prefill built on it
(phase 1 -> la_prefill_front with the gated RMSNorm store), stage by stage against the fp64
oracle on the same inputs each stage received, so that every kernel is held to its own bar:
  rmsnorm_rows: 1 bf16 ulp; projections: the GEMM bar (2^-8 |c| + K 2^-24 sum |a w|);
  gate activations: 2e-6 (1 + |ref|) in fp32; the layer output: the recurrence bars on o, then
  1 bf16 ulp for the gated norm of that o (la_prefill_front without z vs with z).
"""
import math

import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
from linear_attention_chunked_conv1d_gb300.path import Phase1
from tests.helpers import TOL, bf16_ulp_diff, f64, max_abs, rel_frob
import oracle

pytestmark = pytest.mark.gpu


def test_rmsnorm_rows_matches_oracle(cuda):
    g = torch.Generator("cpu")
    g.manual_seed(1)
    for width in (8, 2048, 2056, 8192):
        x = torch.randn(37, width, generator=g).to(torch.bfloat16)
        w = (1 + 0.2 * torch.randn(width, generator=g)).to(torch.bfloat16)
        y = la.rmsnorm_rows(x.to(cuda), w.to(cuda), eps=1e-6)
        torch.cuda.synchronize()
        assert bf16_ulp_diff(y.cpu(), oracle.rmsnorm_rows(f64(x), f64(w), 1e-6)) <= 1, width


def test_gate_activations_match_oracle(cuda):
    g = torch.Generator("cpu")
    g.manual_seed(2)
    ab = (torch.randn(100, 40, generator=g) * 4).to(torch.bfloat16)
    ab[0, :4] = torch.tensor([0.0, 30.0, -30.0, 88.0])
    gg, beta = la.gate_activations(ab.to(cuda), 24)
    torch.cuda.synchronize()
    rg, rb = oracle.gate_activations(f64(ab[:, :24]), f64(ab[:, 24:]))
    for got, ref in ((gg, rg), (beta, rb)):
        err = np.abs(f64(got.cpu()) - ref)
        assert np.all(err <= 2e-6 * (1 + np.abs(ref))), float(err.max())
    assert torch.all(gg <= 0) and torch.all((beta >= 0) & (beta <= 1))


@pytest.mark.parametrize("kda", [False, True])
def test_layer_prefill_from_hidden_rows(cuda, kda):
    """hidden -> norm -> q|k|v, z, a|b projections -> gates -> conv + L2 + recurrence + gated
    RMSNorm, three streams (varlen) with Hk = 1, Hv = 2, d = 128, hidden = 512."""
    gen = torch.Generator("cpu")
    gen.manual_seed(10 + kda)
    lengths = [70, 1, 130]
    T, B, Hk, Hv, D, hid, K = sum(lengths), 3, 1, 2, 128, 512, 4
    cd = 2 * Hk * D + Hv * D
    na = Hv * (D if kda else 1)
    bf = torch.bfloat16
    hidden = torch.randn(T, hid, generator=gen).to(bf)
    norm_w = (1 + 0.1 * torch.randn(hid, generator=gen)).to(bf)
    w_qkv = (torch.randn(cd, hid, generator=gen) / math.sqrt(hid)).to(bf)
    w_z = (torch.randn(Hv * D, hid, generator=gen) / math.sqrt(hid)).to(bf)
    w_ab = (torch.randn(na + Hv, hid, generator=gen) / math.sqrt(hid)).to(bf)
    conv_w = (torch.randn(cd, K, generator=gen) * 0.25).to(bf)
    st0 = torch.randn(B, K - 1, cd, generator=gen).to(bf)
    h0 = torch.randn(B, Hv, D, D, generator=gen) * 0.02
    gn_w = (1 + 0.1 * torch.randn(D, generator=gen)).to(bf)
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)

    class WL:
        variant = "kda" if kda else "gdn"
        d = D
        Hv = 2
    p1 = Phase1(WL, norm_w.to(cuda), w_qkv.to(cuda), w_z.to(cuda), w_ab.to(cuda))
    o1 = p1.run(hidden.to(cuda))
    st, h = st0.clone().to(cuda), h0.clone().to(cuda)
    sp = la.pointer_array([st[s] for s in range(B)])
    hp = la.pointer_array([h[s] for s in range(B)])
    ws = torch.empty(la.prefill_workspace_bytes(B, T, Hk, Hv, D, D, bf), dtype=torch.uint8,
                     device=cuda)
    g = o1["g"].view(T, Hv, D) if kda else o1["g"]
    y = torch.empty(T, Hv, D, dtype=bf, device=cuda)
    la.prefill_front(sp, hp, o1["x"], conv_w.to(cuda), g, o1["beta"], y, cu.to(cuda), Hk=Hk,
                     Hv=Hv, dk=D, dv=D, kda=kda, max_seqlen=max(lengths),
                     z=o1["z"].view(T, Hv, D), norm_w=gn_w.to(cuda), workspace=ws)
    torch.cuda.synchronize()
    assert la.device_status() == 0

    # each stage against the oracle on that stage's own (GPU) inputs
    yn = o1["y"].cpu()
    assert bf16_ulp_diff(yn, oracle.rmsnorm_rows(f64(hidden), f64(norm_w), 1e-6)) <= 1
    for out, wt in ((o1["x"], w_qkv), (o1["z"], w_z), (o1["ab"], w_ab)):
        ref = oracle.linear(f64(yn), f64(wt))
        bound = 2.0 ** -8 * np.abs(ref) + hid * 2.0 ** -24 * (np.abs(f64(yn)) @ np.abs(f64(wt)).T)
        assert np.all(np.abs(f64(out.cpu()) - ref) <= bound)
    rg, rb = oracle.gate_activations(f64(o1["ab"].cpu()[:, :na]), f64(o1["ab"].cpu()[:, na:]))
    assert np.all(np.abs(f64(o1["g"].cpu()) - rg) <= 2e-6 * (1 + np.abs(rg)))
    assert np.all(np.abs(f64(o1["beta"].cpu()) - rb) <= 2e-6 * (1 + np.abs(rb)))
    # the recurrence on the GPU's x, g, beta, then the gated norm of the GPU's o
    xg = f64(o1["x"].cpu())
    q, k, v, ref_st = oracle.front_end(xg, f64(conv_w), f64(st0), cu.numpy(), Hk=Hk, Hv=Hv, dk=D,
                                       dv=D, eps=1e-6, act_dtype="bf16")
    gg = f64(g.cpu())
    ref_o, ref_h = oracle.gated_delta(f64(h0), q, k, v, gg, f64(o1["beta"].cpu()),
                                      cu.numpy().astype(np.int32), scale=1 / math.sqrt(D),
                                      per_channel=kda)
    np.testing.assert_array_equal(f64(st.cpu()), ref_st)
    assert rel_frob(f64(h.cpu()), ref_h) <= TOL["bf16"]["state"]
    # o itself: the same call without z
    st2, h2 = st0.clone().to(cuda), h0.clone().to(cuda)
    o_plain = torch.empty(T, Hv, D, dtype=bf, device=cuda)
    la.prefill_front(la.pointer_array([st2[s] for s in range(B)]),
                     la.pointer_array([h2[s] for s in range(B)]), o1["x"], conv_w.to(cuda), g,
                     o1["beta"], o_plain, cu.to(cuda), Hk=Hk, Hv=Hv, dk=D, dv=D, kda=kda,
                     max_seqlen=max(lengths), workspace=ws)
    torch.cuda.synchronize()
    eo = max_abs(f64(o_plain.cpu()), ref_o)
    assert eo <= TOL["bf16"]["out"], eo
    ref_y = oracle.gated_rmsnorm(f64(o_plain.cpu()), f64(o1["z"].cpu()).reshape(T, Hv, D),
                                 f64(gn_w), 1e-6)
    assert bf16_ulp_diff(y.cpu(), ref_y) <= 1
    print(f"\n[parity] layer from hidden rows kda={kda}: max|o-o_ref| = {eo:.3e}")
