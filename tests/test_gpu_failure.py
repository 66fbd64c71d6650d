"""Failure paths on the GPU, in the forms that fault, trap or hang nothing (GPU).

- A bounded wait that runs out: with LA_DEBUG_STALL=1 the tensor-core kernels make one wait on
  an mbarrier that nothing completes, and LA_WAIT_LIMIT_NS shortens the limit of their waits to
  1 ms. The kernel must give up, drain its own MMAs and copies, free its tensor memory and
  raise LA_DEV_TIMEOUT, which la_device_status() reports; the next call on the same device must
  then run normally and match the oracle.
- Host-side fault injection (LA_FAULT_INJECT=launch): the call returns LA_ERR_CUDA and launches
  nothing, so the caller's buffers keep their contents.

The pages' error convention is that a call the layer cannot run is refused, never half-run
("glm5next_kda/prefill.rs", prefill_with_pad_fill: any other count is refused before a launch).
"""
import math

import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
from linear_attention_chunked_conv1d_gb300.inputs import WORKLOADS, make_inputs, recurrence_inputs
from linear_attention_chunked_conv1d_gb300.path import PrefillPass
from tests.helpers import TOL, f64, max_abs, oracle_recurrence, rel_frob

pytestmark = pytest.mark.gpu

LIMIT_NS = "1000000"  # 1 ms


def _recurrence(cuda, inp, kda=False):
    lengths = inp["lengths"]
    T, B = sum(lengths), len(lengths)
    Hk, Hv, d = inp["q"].shape[1], inp["v"].shape[1], inp["q"].shape[2]
    q, k, v = (inp[n].to(cuda).reshape(T, -1) for n in ("q", "k", "v"))
    g, beta = inp["g"].to(cuda), inp["beta"].to(cuda)
    h = inp["h"].clone().to(cuda)
    out = torch.zeros(T, Hv, d, dtype=torch.bfloat16, device=cuda)
    ptrs = la.pointer_array([h[s] for s in range(B)])
    cu = inp["cu_seqlens"].to(cuda)
    ws = torch.empty(la.prefill_workspace_bytes(B, T, Hk, Hv, d, d, la.LA_BF16),
                     dtype=torch.uint8, device=cuda)
    kw = dict(max_seqlen=max(lengths), Hk=Hk, Hv=Hv, dk=d, dv=d, scale=1.0 / math.sqrt(d),
              workspace=ws)
    if kda:
        la.kda_prefill(ptrs, q, k, v, g, beta, out, cu, **kw)
    else:
        la.gdn_prefill_varlen(ptrs, q, k, v, g, beta, out, cu, **kw)
    torch.cuda.synchronize()
    return out, h


@pytest.mark.parametrize("kda", [False, True])
def test_recurrence_wait_runs_out_then_next_call_is_correct(cuda, monkeypatch, kda):
    inp = recurrence_inputs([300, 64, 1, 129], 2, 4, 128, kda=kda, seed=601)
    assert la.device_status() == 0
    monkeypatch.setenv("LA_DEBUG_STALL", "1")
    monkeypatch.setenv("LA_WAIT_LIMIT_NS", LIMIT_NS)
    _recurrence(cuda, inp, kda)
    st = la.device_status()
    assert st & la.LA_DEV_TIMEOUT, st
    monkeypatch.delenv("LA_DEBUG_STALL")
    monkeypatch.delenv("LA_WAIT_LIMIT_NS")
    # the device is usable: the same call again, every block allocating its tensor memory anew
    out, h = _recurrence(cuda, inp, kda)
    assert la.device_status() == 0
    ref_o, ref_h = oracle_recurrence(inp["h"], inp["q"], inp["k"], inp["v"], inp["g"],
                                     inp["beta"], inp["lengths"], 1.0 / math.sqrt(128), kda)
    tol = TOL["bf16"]
    assert max_abs(f64(out.cpu()), ref_o) <= tol["out"]
    assert rel_frob(f64(h.cpu()), ref_h) <= tol["state"]


def test_fused_front_wait_runs_out_then_next_call_is_correct(cuda, monkeypatch):
    wl = WORKLOADS["kda_varlen_64_h32_d128"].replace(B=3, Hk=2, Hv=2, lengths="list:90,7,200")
    monkeypatch.setenv("LA_DEBUG_STALL", "1")
    monkeypatch.setenv("LA_WAIT_LIMIT_NS", LIMIT_NS)
    inp = make_inputs(wl, device=cuda, seed=602)
    PrefillPass(wl, inp).fused()
    torch.cuda.synchronize()
    assert la.device_status() & la.LA_DEV_TIMEOUT
    monkeypatch.delenv("LA_DEBUG_STALL")
    monkeypatch.delenv("LA_WAIT_LIMIT_NS")
    outs = []
    for mode in ("fused", "split"):  # fresh inputs: the stalled call left its states advanced
        inp = make_inputs(wl, device=cuda, seed=602)
        p = PrefillPass(wl, inp)
        if mode == "fused":
            p.fused()
        else:
            p.front_end()
            p.recurrence()
        torch.cuda.synchronize()
        assert la.device_status() == 0
        outs.append((p.out.clone(), inp["h"].clone(), inp["conv_state"].clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_gemm_wait_runs_out_then_next_call_is_correct(cuda, monkeypatch):
    g = torch.Generator("cpu")
    g.manual_seed(603)
    M, N, K = 1024, 1024, 512  # 32 tiles: the producer fills its ring, then waits
    a = torch.randn(M, K, generator=g).to(torch.bfloat16).to(cuda)
    w = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16).to(cuda)
    c = torch.zeros(M, N, dtype=torch.bfloat16, device=cuda)
    monkeypatch.setenv("LA_DEBUG_STALL", "1")
    monkeypatch.setenv("LA_WAIT_LIMIT_NS", LIMIT_NS)
    la.gemm_bf16(a, w, c)
    torch.cuda.synchronize()
    assert la.device_status() & la.LA_DEV_TIMEOUT
    monkeypatch.delenv("LA_DEBUG_STALL")
    monkeypatch.delenv("LA_WAIT_LIMIT_NS")
    la.gemm_bf16(a, w, c)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    ref = f64(a.cpu()) @ f64(w.cpu()).T
    err = np.abs(f64(c.cpu()) - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -24 * (np.abs(f64(a.cpu())) @ np.abs(f64(w.cpu())).T))


def test_injected_launch_failure_touches_nothing(cuda, monkeypatch):
    inp = recurrence_inputs([40, 3], 1, 2, 128, seed=604)
    x = torch.randn(43, 512, device=cuda).to(torch.bfloat16)
    out = torch.full_like(x, 7.0)
    cs = torch.full((2, 3, 512), 5.0, dtype=torch.bfloat16, device=cuda)
    ptrs = la.pointer_array([cs[0], cs[1]])
    w = torch.randn(512, 4, device=cuda).to(torch.bfloat16)
    cu = inp["cu_seqlens"].to(cuda)
    monkeypatch.setenv("LA_FAULT_INJECT", "launch")
    with pytest.raises(la.LinAttnError) as ei:
        la.conv1d_silu_prefill_varlen(ptrs, x, w, out, cu)
    assert ei.value.code == la.LA_ERR_CUDA and "injected" in str(ei.value)
    monkeypatch.delenv("LA_FAULT_INJECT")
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(cs == 5.0)
    la.conv1d_silu_prefill_varlen(ptrs, x, w, out, cu)  # and without injection it runs
    torch.cuda.synchronize()
    assert not torch.all(out == 7.0)
