"""GPU parity of the one-launch layer prefill (la_prefill_front: conv1d + SiLU + q|k L2 +
recurrence, the conv output kept on chip) against the fp64 oracle, and bit-for-bit against the
separate calls (la_conv1d_silu_l2_prefill, then the recurrence call) on the same inputs.

Cases: GDN batched and varlen, KDA single stream and varlen, GQA groups of 1, 2 and 4, streams
of length 0, 1, 2 (shorter than the conv window), 64, 65 and several chunks, conv kernels 1..4
with and without bias, pad_fill 0 / 1e3 / NaN, and the argument checks.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
from tests.helpers import TOL, f64, max_abs, rel_frob
import oracle

pytestmark = pytest.mark.gpu

D = 128


def make_case(lengths, Hk, Hv, K, kda, seed, bias=False):
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    T, B = sum(lengths), len(lengths)
    cd = 2 * Hk * D + Hv * D
    bf = torch.bfloat16
    x = torch.randn(T, cd, generator=g).to(bf)
    w = (torch.randn(cd, K, generator=g) * 0.25).to(bf)
    b = (torch.randn(cd, generator=g) * 0.5).to(bf) if bias else None
    st = torch.randn(B, max(K - 1, 1), cd, generator=g).to(bf)[:, :K - 1].contiguous()
    h = torch.randn(B, Hv, D, D, generator=g) * 0.02
    gshape = (T, Hv, D) if kda else (T, Hv)
    gate = -torch.nn.functional.softplus(torch.randn(*gshape, generator=g))
    beta = torch.sigmoid(torch.randn(T, Hv, generator=g))
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)
    return dict(lengths=list(lengths), x=x, w=w, b=b, st=st, h=h, g=gate, beta=beta, cu=cu,
                Hk=Hk, Hv=Hv, K=K, kda=kda)


def run_fused(cuda, c, *, batched=False, pad_fill=0.0):
    lengths, Hk, Hv, K = c["lengths"], c["Hk"], c["Hv"], c["K"]
    T, B = sum(lengths), len(lengths)
    st = c["st"].clone().to(cuda)
    h = c["h"].clone().to(cuda)
    out = torch.full((T, Hv, D), 5.0, dtype=torch.bfloat16, device=cuda)
    sp = la.pointer_array([st[s] for s in range(B)]) if K > 1 else None
    hp = la.pointer_array([h[s] for s in range(B)])
    ws = torch.empty(la.prefill_workspace_bytes(B, T, Hk, Hv, D, D, torch.bfloat16),
                     dtype=torch.uint8, device=cuda)
    la.prefill_front(sp, hp, c["x"].to(cuda), c["w"].to(cuda), c["g"].to(cuda),
                     c["beta"].to(cuda), out, None if batched else c["cu"].to(cuda), B=B, Hk=Hk,
                     Hv=Hv, dk=D, dv=D, kda=c["kda"],
                     conv_bias=None if c["b"] is None else c["b"].to(cuda),
                     max_seqlen=max(lengths), pad_fill=pad_fill, workspace=ws)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    return out.cpu(), h.cpu(), st.cpu()


def run_separate(cuda, c):
    """The same layer through the separate calls: fused conv + L2, then the recurrence."""
    lengths, Hk, Hv, K = c["lengths"], c["Hk"], c["Hv"], c["K"]
    T, B = sum(lengths), len(lengths)
    st = c["st"].clone().to(cuda)
    h = c["h"].clone().to(cuda)
    x = c["x"].to(cuda)
    cu = c["cu"].to(cuda)
    conv_out = torch.empty_like(x)
    sp = la.pointer_array([st[s] for s in range(B)]) if K > 1 else \
        torch.zeros(B, dtype=torch.int64, device=cuda)
    la.conv1d_silu_l2_prefill(sp, x, c["w"].to(cuda), conv_out, cu, l2_heads=2 * Hk,
                              head_dim=D, eps=1e-6,
                              bias=None if c["b"] is None else c["b"].to(cuda))
    hk = Hk * D
    q, k, v = conv_out[:, :hk], conv_out[:, hk:2 * hk], conv_out[:, 2 * hk:]
    out = torch.empty(T, Hv, D, dtype=torch.bfloat16, device=cuda)
    hp = la.pointer_array([h[s] for s in range(B)])
    ws = torch.empty(la.prefill_workspace_bytes(B, T, Hk, Hv, D, D, torch.bfloat16),
                     dtype=torch.uint8, device=cuda)
    if c["kda"]:
        la.kda_prefill(hp, q, k, v, c["g"].to(cuda), c["beta"].to(cuda), out, cu, Hk=Hk, Hv=Hv,
                       dk=D, dv=D, max_seqlen=max(lengths), workspace=ws)
    else:
        la.gdn_prefill_varlen(hp, q, k, v, c["g"].to(cuda), c["beta"].to(cuda), out, cu,
                              max_seqlen=max(lengths), Hk=Hk, Hv=Hv, dk=D, dv=D, workspace=ws)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    return out.cpu(), h.cpu(), st.cpu()


def check_oracle(c, out, h, st):
    lengths, Hk, Hv = c["lengths"], c["Hk"], c["Hv"]
    cu = np.asarray(c["cu"].numpy())
    q, k, v, ref_st = oracle.front_end(f64(c["x"]), f64(c["w"]), f64(c["st"]), cu, Hk=Hk, Hv=Hv,
                                       dk=D, dv=D, eps=1e-6, act_dtype="bf16",
                                       bias=None if c["b"] is None else f64(c["b"]))
    ref_o, ref_h = oracle.gated_delta(f64(c["h"]), q, k, v, f64(c["g"]), f64(c["beta"]),
                                      cu.astype(np.int32), scale=1.0 / math.sqrt(D),
                                      per_channel=c["kda"])
    if c["K"] > 1:
        np.testing.assert_array_equal(f64(st), ref_st)
    eo = max_abs(f64(out), ref_o)
    eh = rel_frob(f64(h), ref_h)
    print(f"\n[parity] fused prefill {'KDA' if c['kda'] else 'GDN'} Hk={Hk} Hv={Hv} "
          f"K={c['K']} lengths={lengths}: max|o-o_ref| = {eo:.3e}, state rel.Frobenius = {eh:.3e}")
    assert eo <= TOL["bf16"]["out"]
    assert eh <= TOL["bf16"]["state"]


CASES = {
    "gdn_varlen_gqa2": dict(lengths=[1, 2, 0, 64, 65, 130, 200, 3], Hk=2, Hv=4, K=4, kda=False),
    "gdn_gqa1_bias_k3": dict(lengths=[150, 7, 64], Hk=2, Hv=2, K=3, kda=False, bias=True),
    "gdn_k2": dict(lengths=[1, 90], Hk=1, Hv=2, K=2, kda=False),
    "gdn_k1": dict(lengths=[70, 5], Hk=1, Hv=1, K=1, kda=False),
    "kda_single": dict(lengths=[150], Hk=2, Hv=2, K=4, kda=True),
    "kda_varlen_gqa4": dict(lengths=[70, 1, 129, 0, 5], Hk=1, Hv=4, K=4, kda=True),
    "kda_bias_k4": dict(lengths=[33, 100], Hk=1, Hv=1, K=4, kda=True, bias=True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_front_equals_separate_calls_and_oracle(cuda, name):
    spec = dict(CASES[name])
    c = make_case(spec.pop("lengths"), spec.pop("Hk"), spec.pop("Hv"), spec.pop("K"),
                  spec.pop("kda"), seed=zlib.crc32(name.encode()) % 1000, **spec)
    fo, fh, fs = run_fused(cuda, c)
    so, sh, ss = run_separate(cuda, c)
    assert torch.equal(fo, so), "outputs differ from the separate calls"
    assert torch.equal(fh, sh), "h states differ from the separate calls"
    assert torch.equal(fs, ss), "conv states differ from the separate calls"
    check_oracle(c, fo, fh, fs)


def test_front_batched_equals_varlen(cuda):
    c = make_case([130, 130, 130], 2, 2, 4, False, seed=5)
    a = run_fused(cuda, c, batched=True)
    b = run_fused(cuda, c, batched=False)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    check_oracle(c, *a)


@pytest.mark.parametrize("kda", [False, True])
def test_front_pad_fill_invariance_bitwise(cuda, kda):
    """KDA masks the pad rows by select; GDN ignores pad_fill (zero pad rows)."""
    c = make_case([45, 130, 1], 1, 2, 4, kda, seed=11)
    ref = run_fused(cuda, c, pad_fill=0.0)
    for pf in (1e3, float("nan")):
        got = run_fused(cuda, c, pad_fill=pf)
        for u, v in zip(ref, got):
            assert torch.equal(u, v)


def test_front_zero_length_stream_keeps_states(cuda):
    c = make_case([0, 10, 0], 1, 2, 4, False, seed=2)
    out, h, st = run_fused(cuda, c)
    assert torch.equal(h[0], c["h"][0]) and torch.equal(h[2], c["h"][2])
    assert torch.equal(st[0], c["st"][0]) and torch.equal(st[2], c["st"][2])
    check_oracle(c, out, h, st)


def test_front_refusals_leave_buffers_untouched(cuda):
    c = make_case([10, 20], 1, 2, 4, False, seed=3)
    T = 30
    x = c["x"].to(cuda)
    w = c["w"].to(cuda)
    st = c["st"].clone().to(cuda)
    h = c["h"].clone().to(cuda)
    out = torch.full((T, 2, D), 5.0, dtype=torch.bfloat16, device=cuda)
    sp = la.pointer_array([st[s] for s in range(2)])
    hp = la.pointer_array([h[s] for s in range(2)])
    g, beta, cu = c["g"].to(cuda), c["beta"].to(cuda), c["cu"].to(cuda)
    ws = torch.empty(la.prefill_workspace_bytes(2, T, 1, 2, D, D, torch.bfloat16),
                     dtype=torch.uint8, device=cuda)
    common = dict(Hk=1, Hv=2, dk=D, dv=D, kda=False, max_seqlen=20)
    with pytest.raises(la.LinAttnError) as ei:   # too small a workspace
        la.prefill_front(sp, hp, x, w, g, beta, out, cu, workspace=ws[:16], **common)
    assert ei.value.code == la.LA_ERR_ARG
    with pytest.raises(la.LinAttnError) as ei:   # head dim outside the tensor-core path
        la.prefill_front(sp, hp, x, w, g, beta, out, cu, workspace=ws,
                         **{**common, "dk": 64, "dv": 64})
    assert ei.value.code == la.LA_ERR_UNSUPPORTED
    with pytest.raises(la.LinAttnError) as ei:   # fp32 activations
        la.prefill_front(sp, hp, x.float(), w.float(), g, beta, out.float(), cu, workspace=ws,
                         **common)
    assert ei.value.code == la.LA_ERR_UNSUPPORTED
    with pytest.raises(la.LinAttnError) as ei:   # token count above max_tokens
        la.prefill_front(sp, hp, x, w, g, beta, out, cu, workspace=ws, max_tokens=T - 1,
                         **common)
    assert ei.value.code == la.LA_ERR_COUNT
    with pytest.raises(la.LinAttnError) as ei:   # batched: total not a multiple of B
        la.prefill_front(sp, hp, x[:29], w, g, beta, out, None, B=2, workspace=ws,
                         **{**common, "max_seqlen": None})
    assert ei.value.code == la.LA_ERR_ARG
    torch.cuda.synchronize()
    assert torch.all(out.cpu() == 5.0)
    assert torch.equal(h.cpu(), c["h"]) and torch.equal(st.cpu(), c["st"])


def test_front_many_short_streams(cuda):
    """2500 streams (many empty or shorter than the conv window, a few several chunks long):
    the stream order kernel past 1024 streams, the persistent scheduler over 5000 units, the
    conv-state reader counts of 2500 (stream, k-head) pairs."""
    g = torch.Generator("cpu")
    g.manual_seed(77)
    lengths = torch.randint(0, 6, (2500,), generator=g).tolist()
    for i in (5, 900, 2400):
        lengths[i] = 150 + i % 50
    c = make_case(lengths, 1, 2, 4, False, seed=78)
    fo, fh, fs = run_fused(cuda, c)
    so, sh, ss = run_separate(cuda, c)
    assert torch.equal(fo, so) and torch.equal(fh, sh) and torch.equal(fs, ss)
    check_oracle(c, fo, fh, fs)
