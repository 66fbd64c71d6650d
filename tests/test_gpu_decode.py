"""GPU parity of the decode step (la_decode_step: one new token per stream on the carried conv
and h states) against the fp64 oracle: single steps, a run of steps that must equal the prefill
of the same tokens, a prefill followed by decode steps, the full-size decode workloads, and the
argument checks. The oracle is the same per-token recurrence and conv as for the prefill.
"""
import math

import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
from linear_attention_chunked_conv1d_gb300.inputs import DECODE_WORKLOADS, make_inputs
from linear_attention_chunked_conv1d_gb300.path import DecodeStep, PrefillPass
from tests.helpers import TOL, f64, max_abs, rel_frob
import oracle

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_seq(B, T, Hk, Hv, d, K, kda, dtype, seed):
    """T tokens for each of B streams, stored stream-major [B][T][...]."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    cd = 2 * Hk * d + Hv * d
    act = DT[dtype]
    x = torch.randn(B, T, cd, generator=g).to(act)
    w = (torch.randn(cd, K, generator=g) * 0.25).to(act)
    st = torch.randn(B, max(K - 1, 1), cd, generator=g).to(act)[:, :K - 1].contiguous()
    h = torch.randn(B, Hv, d, d, generator=g) * 0.02
    gshape = (B, T, Hv, d) if kda else (B, T, Hv)
    gate = -torch.nn.functional.softplus(torch.randn(*gshape, generator=g))
    beta = torch.sigmoid(torch.randn(B, T, Hv, generator=g))
    return dict(x=x, w=w, st=st, h=h, g=gate, beta=beta, B=B, T=T, Hk=Hk, Hv=Hv, d=d, K=K,
                kda=kda, dtype=dtype)


def oracle_seq(c, T=None):
    """Oracle over the first T tokens of every stream (the prefill definition)."""
    B, d = c["B"], c["d"]
    T = c["T"] if T is None else T
    x = f64(c["x"][:, :T]).reshape(B * T, -1)
    cu = np.arange(0, B * T + 1, T)
    q, k, v, st = oracle.front_end(x, f64(c["w"]), f64(c["st"]), cu, Hk=c["Hk"], Hv=c["Hv"],
                                   dk=d, dv=d, eps=1e-6, act_dtype=c["dtype"])
    g = f64(c["g"][:, :T]).reshape(B * T, *c["g"].shape[2:])
    beta = f64(c["beta"][:, :T]).reshape(B * T, -1)
    o, h = oracle.gated_delta(f64(c["h"]), q, k, v, g, beta, cu.astype(np.int32),
                              scale=1.0 / math.sqrt(d), per_channel=c["kda"])
    return o.reshape(B, T, c["Hv"], d), h, st


class Dev:
    """Device copies of one case's states and the decode call on token t of every stream."""

    def __init__(self, cuda, c):
        self.c = c
        B, d = c["B"], c["d"]
        self.st = c["st"].clone().to(cuda)
        self.h = c["h"].clone().to(cuda)
        self.sp = la.pointer_array([self.st[s] for s in range(B)]) if c["K"] > 1 else None
        self.hp = la.pointer_array([self.h[s] for s in range(B)])
        self.w = c["w"].to(cuda)
        self.ws = torch.empty(la.decode_workspace_bytes(B, c["Hk"], c["Hv"], d, d, DT[c["dtype"]]),
                              dtype=torch.uint8, device=cuda)
        self.cuda = cuda

    def step(self, t):
        c = self.c
        out = torch.full((c["B"], c["Hv"], c["d"]), 7.0, dtype=DT[c["dtype"]], device=self.cuda)
        la.decode_step(self.sp, self.hp, c["x"][:, t].contiguous().to(self.cuda), self.w,
                       c["g"][:, t].contiguous().to(self.cuda),
                       c["beta"][:, t].contiguous().to(self.cuda), out, Hk=c["Hk"], Hv=c["Hv"],
                       dk=c["d"], dv=c["d"], kda=c["kda"], workspace=self.ws)
        return out


def check(c, got_o, got_h, got_st, ref_o, ref_h, ref_st, label):
    tol = TOL[c["dtype"]]
    eo = max_abs(f64(got_o), ref_o)
    eh = rel_frob(f64(got_h), ref_h)
    print(f"\n[parity] decode {label}: max|o-o_ref| = {eo:.3e}, state rel.Frobenius = {eh:.3e}")
    assert eo <= tol["out"], eo
    assert eh <= tol["state"], eh
    if c["K"] > 1:
        np.testing.assert_array_equal(f64(got_st), ref_st)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kda", [False, True])
def test_decode_steps_equal_prefill_of_the_same_tokens(cuda, dtype, d, kda):
    c = make_seq(B=5, T=6, Hk=1, Hv=2 if kda else 4, d=d, K=4, kda=kda, dtype=dtype,
                 seed=d + 7 * kda + (dtype == "bf16"))
    dev = Dev(cuda, c)
    outs = [dev.step(t) for t in range(c["T"])]
    torch.cuda.synchronize()
    assert la.device_status() == 0
    got_o = torch.stack([o.cpu() for o in outs], dim=1)
    ref_o, ref_h, ref_st = oracle_seq(c)
    check(c, got_o, dev.h.cpu(), dev.st.cpu(), ref_o, ref_h, ref_st,
          f"{dtype} d={d} kda={kda} 6 steps")


@pytest.mark.parametrize("K", [1, 2, 3])
def test_decode_short_conv_kernels(cuda, K):
    c = make_seq(B=3, T=3, Hk=2, Hv=2, d=128, K=K, kda=False, dtype="bf16", seed=40 + K)
    dev = Dev(cuda, c)
    outs = [dev.step(t) for t in range(c["T"])]
    torch.cuda.synchronize()
    got_o = torch.stack([o.cpu() for o in outs], dim=1)
    ref_o, ref_h, ref_st = oracle_seq(c)
    check(c, got_o, dev.h.cpu(), dev.st.cpu(), ref_o, ref_h, ref_st, f"K={K}")


@pytest.mark.parametrize("kda", [False, True])
def test_prefill_then_decode(cuda, kda):
    """Prefill the first 70 tokens (the bench's path), then decode three more."""
    B, T0, T = 3, 70, 73
    c = make_seq(B=B, T=T, Hk=2, Hv=4, d=128, K=4, kda=kda, dtype="bf16", seed=90 + kda)
    dev = Dev(cuda, c)
    x = c["x"][:, :T0].reshape(B * T0, -1).to(cuda)
    gg = c["g"][:, :T0].reshape(B * T0, *c["g"].shape[2:]).to(cuda)
    bb = c["beta"][:, :T0].reshape(B * T0, -1).to(cuda)
    out0 = torch.empty(B * T0, c["Hv"], 128, dtype=torch.bfloat16, device=cuda)
    ws = torch.empty(la.prefill_workspace_bytes(B, B * T0, 2, 4, 128, 128, torch.bfloat16),
                     dtype=torch.uint8, device=cuda)
    la.prefill_front(dev.sp, dev.hp, x, dev.w, gg, bb, out0, None, B=B, Hk=2, Hv=4, dk=128,
                     dv=128, kda=kda, workspace=ws)
    outs = [dev.step(t) for t in range(T0, T)]
    torch.cuda.synchronize()
    assert la.device_status() == 0
    ref_o, ref_h, ref_st = oracle_seq(c)
    got_o = torch.stack([o.cpu() for o in outs], dim=1)
    check(c, got_o, dev.h.cpu(), dev.st.cpu(), ref_o[:, T0:], ref_h, ref_st, f"kda={kda} after prefill")
    assert max_abs(f64(out0.cpu()).reshape(B, T0, 4, 128), ref_o[:, :T0]) <= TOL["bf16"]["out"]


@pytest.mark.parametrize("name", list(DECODE_WORKLOADS))
def test_decode_workload_full_size(cuda, name):
    """The decode step the bench times, at its full size, against the oracle on every unit."""
    wl = DECODE_WORKLOADS[name]
    inp = make_inputs(wl, device="cpu", seed=0)
    ref = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in inp.items()}
    dinp = {k: (v.to(cuda) if torch.is_tensor(v) else v) for k, v in inp.items()}
    step = DecodeStep(wl, dinp)
    step.run()
    torch.cuda.synchronize()
    assert la.device_status() == 0
    cu = np.arange(wl.B + 1)
    q, k, v, st = oracle.front_end(f64(ref["x"]), f64(ref["conv_w"]), f64(ref["conv_state"]), cu,
                                   Hk=wl.Hk, Hv=wl.Hv, dk=wl.d, dv=wl.d, eps=1e-6,
                                   act_dtype=wl.dtype)
    o, h = oracle.gated_delta(f64(ref["h"]), q, k, v, f64(ref["g"]), f64(ref["beta"]),
                              cu.astype(np.int32), scale=1.0 / math.sqrt(wl.d),
                              per_channel=wl.variant == "kda")
    c = dict(dtype=wl.dtype, K=wl.conv_kernel)
    check(c, step.out.cpu(), dinp["h"].cpu(), dinp["conv_state"].cpu(), o, h, st, name)


def test_decode_refusals_leave_buffers_untouched(cuda):
    c = make_seq(B=2, T=1, Hk=1, Hv=2, d=128, K=4, kda=False, dtype="bf16", seed=3)
    dev = Dev(cuda, c)
    x = c["x"][:, 0].contiguous().to(cuda)
    g, beta = c["g"][:, 0].contiguous().to(cuda), c["beta"][:, 0].contiguous().to(cuda)
    out = torch.full((2, 2, 128), 7.0, dtype=torch.bfloat16, device=cuda)
    common = dict(Hk=1, Hv=2, dk=128, dv=128, kda=False)
    cases = [(dict(workspace=dev.ws[:16]), la.LA_ERR_ARG),
             (dict(workspace=dev.ws, max_streams=1), la.LA_ERR_COUNT),
             (dict(workspace=dev.ws, dk=96, dv=96), la.LA_ERR_UNSUPPORTED),
             (dict(workspace=dev.ws, Hk=2, Hv=3), la.LA_ERR_ARG)]
    for kw, code in cases:
        with pytest.raises(la.LinAttnError) as ei:
            la.decode_step(dev.sp, dev.hp, x, dev.w, g, beta, out, **{**common, **kw})
        assert ei.value.code == code, (kw, ei.value)
    torch.cuda.synchronize()
    assert torch.all(out.cpu() == 7.0)
    assert torch.equal(dev.h.cpu(), c["h"]) and torch.equal(dev.st.cpu(), c["st"])
