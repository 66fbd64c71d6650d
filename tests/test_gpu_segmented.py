"""GPU parity of the chunk-parallel scan of one long stream (la_prefill_segmented: segments run
side by side, joined through their state transitions) against the fp64 oracle and against the
plain one-block-per-unit call: GDN and KDA, 2..5 segments, lengths that leave ragged last
segments or fewer chunks than segments, segments = 1 (bit for bit the plain call), and the full
KDA T = 4096 workload. Bars: the recurrence bars (outputs 2e-3 absolute, states 1e-3 relative
Frobenius); the extra roundings of the join (the outputs of a segment are rounded to bf16 once
before the correction and once after) stay far inside them.
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


def run(cuda, inp, Hk, Hv, kda, segments):
    T = inp["lengths"][0]
    q, k, v = (inp[n].to(cuda).reshape(T, -1) for n in ("q", "k", "v"))
    h = inp["h"].clone().to(cuda)
    out = torch.full((T, Hv, 128), 3.0, dtype=torch.bfloat16, device=cuda)
    ws = torch.empty(la.prefill_segmented_workspace_bytes(T, Hv, segments), dtype=torch.uint8,
                     device=cuda)
    la.prefill_segmented(la.pointer_array([h[0]]), q, k, v, inp["g"].to(cuda),
                         inp["beta"].to(cuda), out, Hk=Hk, Hv=Hv, dk=128, dv=128, kda=kda,
                         segments=segments, workspace=ws)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    return out.cpu(), h.cpu()


def run_plain(cuda, inp, Hk, Hv, kda):
    T = inp["lengths"][0]
    q, k, v = (inp[n].to(cuda).reshape(T, -1) for n in ("q", "k", "v"))
    h = inp["h"].clone().to(cuda)
    out = torch.empty(T, Hv, 128, dtype=torch.bfloat16, device=cuda)
    ws = torch.empty(la.prefill_workspace_bytes(1, T, Hk, Hv, 128, 128, torch.bfloat16),
                     dtype=torch.uint8, device=cuda)
    ptrs = la.pointer_array([h[0]])
    if kda:
        la.kda_prefill(ptrs, q, k, v, inp["g"].to(cuda), inp["beta"].to(cuda), out, Hk=Hk, Hv=Hv,
                       dk=128, dv=128, workspace=ws)
    else:
        la.gdn_prefill_batched(ptrs, q, k, v, inp["g"].to(cuda), inp["beta"].to(cuda), out, B=1,
                               T=T, Hk=Hk, Hv=Hv, dk=128, dv=128, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu(), h.cpu()


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("T,segments", [(1000, 2), (1000, 3), (300, 5), (130, 4), (640, 2)])
def test_segmented_matches_oracle_and_plain(cuda, kda, T, segments):
    Hk, Hv = 2, 4
    inp = recurrence_inputs([T], Hk, Hv, 128, kda=kda, seed=T + segments + 7 * kda)
    o, h = run(cuda, inp, Hk, Hv, kda, segments)
    ref_o, ref_h = oracle_recurrence(inp["h"], inp["q"], inp["k"], inp["v"], inp["g"],
                                     inp["beta"], [T], 1 / math.sqrt(128), kda)
    eo, eh = max_abs(f64(o), ref_o), rel_frob(f64(h), ref_h)
    po, ph = run_plain(cuda, inp, Hk, Hv, kda)
    print(f"\n[parity] segmented kda={kda} T={T} S={segments}: max|o-o_ref| = {eo:.3e}, state "
          f"rel.Frobenius = {eh:.3e} (plain call: {max_abs(f64(po), ref_o):.3e}, "
          f"{rel_frob(f64(ph), ref_h):.3e})")
    assert eo <= TOL["bf16"]["out"] and eh <= TOL["bf16"]["state"]


def test_one_segment_is_the_plain_call(cuda):
    inp = recurrence_inputs([333], 1, 2, 128, kda=True, seed=3)
    a = run(cuda, inp, 1, 2, True, 1)
    b = run_plain(cuda, inp, 1, 2, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_segmented_full_kda_t4096(cuda):
    """The KDA T = 4096, 32-head workload (front end as the bench runs it), recurrence through
    the segmented scan with 2 segments, against the oracle on every head."""
    wl = WORKLOADS["kda_t4096_h32_d128"]
    inp = make_inputs(wl, device="cpu", seed=0)
    ref_in = {k_: (v_.clone() if torch.is_tensor(v_) else v_) for k_, v_ in inp.items()}
    dinp = {k_: (v_.to(cuda) if torch.is_tensor(v_) else v_) for k_, v_ in inp.items()}
    p = PrefillPass(wl, dinp)
    p.front_end()
    p.recurrence_segmented(2)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    import oracle
    T = 4096
    cu = np.array([0, T])
    q, k, v, _ = oracle.front_end(f64(ref_in["x"]), f64(ref_in["conv_w"]),
                                  f64(ref_in["conv_state"]), cu, Hk=32, Hv=32, dk=128, dv=128,
                                  eps=1e-6, act_dtype="bf16")
    ref_o, ref_h = oracle.gated_delta(f64(ref_in["h"]), q, k, v, f64(ref_in["g"]),
                                      f64(ref_in["beta"]), cu.astype(np.int32),
                                      scale=1 / math.sqrt(128), per_channel=True)
    eo, eh = max_abs(f64(p.out.cpu()), ref_o), rel_frob(f64(dinp["h"].cpu()), ref_h)
    print(f"\n[parity] segmented kda_t4096_h32_d128 S=2: max|o-o_ref| = {eo:.3e}, "
          f"state rel.Frobenius = {eh:.3e}")
    assert eo <= TOL["bf16"]["out"] and eh <= TOL["bf16"]["state"]
