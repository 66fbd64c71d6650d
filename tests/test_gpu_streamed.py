"""The pipelined host-to-host driver (path.StreamedPrefill: copies of neighbouring steps overlap
each step's compute on three streams) gives, bit for bit, what the same steps give run one after
another on one stream: outputs of every step, final conv and h states. Checked for the two-launch
and fused paths over four steps with different inputs per step.
"""
import pytest
import torch

from linear_attention_chunked_conv1d_gb300.inputs import WORKLOADS, make_inputs
from linear_attention_chunked_conv1d_gb300.path import PrefillPass, StreamedPrefill

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["split", "fused"])
def test_streamed_equals_sequential(cuda, mode):
    wl = WORKLOADS["gdn_varlen_32_hk16_hv32_d128"].replace(B=3, Hk=2, Hv=4,
                                                           lengths="list:70,1,130")
    steps = 4
    hosts = [make_inputs(wl, device="cpu", seed=s) for s in range(steps)]
    base = make_inputs(wl, device=cuda, seed=100)
    # sequential reference on one stream
    ref_state = {k: v.clone() for k, v in base.items() if torch.is_tensor(v)}
    ref_in = dict(base, **ref_state)
    p = PrefillPass(wl, ref_in)
    ref_outs = []
    for s in range(steps):
        for name in ("x", "g", "beta"):
            ref_in[name].copy_(hosts[s][name].to(cuda))
        (p.fused() if mode == "fused" else p.run_unfused())
        ref_outs.append(p.out.cpu().clone())
    torch.cuda.synchronize()
    # pipelined
    sp_in = dict(base)
    sp_in["conv_state"], sp_in["h"] = base["conv_state"].clone(), base["h"].clone()
    sp = StreamedPrefill(wl, sp_in, mode=mode)
    outs = [torch.empty(ref_outs[0].shape, dtype=ref_outs[0].dtype).pin_memory() for _ in range(steps)]
    pinned = [{n: hosts[s][n].pin_memory() for n in ("x", "g", "beta")} for s in range(steps)]
    for s in range(steps):
        sp.step(s, pinned[s]["x"], pinned[s]["g"], pinned[s]["beta"], outs[s])
    sp.finish()
    torch.cuda.synchronize()
    for s in range(steps):
        assert torch.equal(outs[s], ref_outs[s]), s
    assert torch.equal(sp_in["h"], ref_in["h"]) and torch.equal(sp_in["conv_state"], ref_in["conv_state"])
