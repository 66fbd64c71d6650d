"""The no-allocation GDN entry point against the workspace one (GPU).

Some callers cannot allocate device memory when they run this layer: an engine that has
already handed all device memory to its own allocator, or a plugin interface with a fixed
signature and no slot for a workspace. la_gdn_prefill_varlen_noalloc serves them from a
fixed scratch array inside the library. This file is collected last on purpose, so that a
failure here cannot hide the results of the other tests.
"""
import math

import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
import oracle
from linear_attention_chunked_conv1d_gb300.inputs import recurrence_inputs
from tests.helpers import TOL, f64, max_abs, rel_frob

pytestmark = pytest.mark.gpu


def _run(cuda, inp, noalloc):
    lengths = inp["lengths"]
    T, B = sum(lengths), len(lengths)
    Hk, Hv, d = inp["q"].shape[1], inp["v"].shape[1], inp["q"].shape[2]
    q, k, v = (inp[n].to(cuda).reshape(T, -1) for n in ("q", "k", "v"))
    g, beta = inp["g"].to(cuda), inp["beta"].to(cuda)
    h = inp["h"].clone().to(cuda)
    out = torch.zeros(T, Hv, d, dtype=torch.bfloat16, device=cuda)
    ptrs = la.pointer_array([h[s] for s in range(B)])
    cu = inp["cu_seqlens"].to(cuda)
    kw = dict(max_seqlen=max(lengths), Hk=Hk, Hv=Hv, dk=d, dv=d, scale=1.0 / math.sqrt(d))
    if noalloc:
        la.gdn_prefill_varlen_noalloc(ptrs, q, k, v, g, beta, out, cu, **kw)
    else:
        ws = torch.empty(la.prefill_workspace_bytes(B, T, Hk, Hv, d, d, la.LA_BF16),
                         dtype=torch.uint8, device=cuda)
        la.gdn_prefill_varlen(ptrs, q, k, v, g, beta, out, cu, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    return out.cpu(), h.cpu()


def _oracle(inp):
    lengths = inp["lengths"]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    d = inp["q"].shape[2]
    return oracle.gated_delta(f64(inp["h"]), f64(inp["q"]), f64(inp["k"]), f64(inp["v"]),
                              f64(inp["g"]), f64(inp["beta"]), cu, scale=1.0 / math.sqrt(d))


def test_noalloc_matches_workspace_call_twice_in_a_row(cuda):
    """Same kernel, same inputs: the no-allocation call gives the bits of the workspace call.
    The calls run back to back on the shared scratch; the first case has 200 streams, whose
    stream order fills the bytes where the later, smaller calls keep their unit counter, so
    those calls only work if each call re-initialises what it reads."""
    r = np.random.default_rng(500)
    many = [int(v) for v in r.integers(0, 40, size=200)]
    cases = [recurrence_inputs(many, 1, 2, 128, seed=500),
             recurrence_inputs([130, 1, 64, 0, 257], 2, 4, 128, seed=501),
             recurrence_inputs([70, 300], 1, 2, 128, seed=502)]
    for i, inp in enumerate(cases):
        o_ref, h_ref = _run(cuda, inp, noalloc=False)
        o_na, h_na = _run(cuda, inp, noalloc=True)
        assert torch.equal(o_na, o_ref), i
        assert torch.equal(h_na, h_ref), i
        if i == 1:  # and once against the oracle directly
            ref_o, ref_h = _oracle(inp)
            tol = TOL["bf16"]
            assert max_abs(f64(o_na), ref_o) <= tol["out"]
            assert rel_frob(f64(h_na), ref_h) <= tol["state"]


def test_noalloc_accepts_the_stream_limit(cuda):
    """4096 one-token streams, the most the fixed scratch serves, then a 3-stream call."""
    for lengths in ([1] * 4096, [5, 9, 2]):
        inp = recurrence_inputs(lengths, 1, 1, 128, seed=503)
        o_ref, h_ref = _run(cuda, inp, noalloc=False)
        o_na, h_na = _run(cuda, inp, noalloc=True)
        assert torch.equal(o_na, o_ref) and torch.equal(h_na, h_ref)


def test_noalloc_refuses_too_many_streams(cuda):
    B = 4097
    x = torch.zeros(B, 128, dtype=torch.bfloat16, device=cuda)
    g = torch.zeros(B, 1, device=cuda)
    cu = torch.arange(B + 1, dtype=torch.int32, device=cuda)
    ptrs = torch.zeros(B, dtype=torch.int64, device=cuda)
    with pytest.raises(la.LinAttnError) as ei:
        la.gdn_prefill_varlen_noalloc(ptrs, x, x, x, g, g, x.view(B, 1, 128), cu, max_seqlen=1,
                                      Hk=1, Hv=1, dk=128, dv=128)
    assert ei.value.code == la.LA_ERR_UNSUPPORTED
    assert "4096" in la.last_error()
