"""Full-size workloads on the GPU, through every public path the bench can report (PrefillPass:
the one-launch la_prefill_front where it applies, the two-launch path — fused conv1d+SiLU+L2,
then the recurrence — and, for a single stream, the segmented recurrence), checked against the
oracle on sampled (stream, v-head) units: every sampled unit's outputs, final state and the
stream's conv state. Units are independent, so a sample is checked exactly as the whole would
be. The sample holds the shortest stream, whose units the longest-first scheduler hands out
last (after every block has walked many units), the longest and the median one.
"""
import math

import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
from linear_attention_chunked_conv1d_gb300.inputs import WORKLOADS, make_inputs
from linear_attention_chunked_conv1d_gb300.path import PrefillPass
from tests.helpers import TOL, f64, max_abs, oracle_front, oracle_recurrence, rel_frob

pytestmark = pytest.mark.gpu


def sample_units(wl, lengths):
    if wl.B == 1:
        streams = [0]
    else:
        order = np.argsort(lengths)
        streams = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2])})
    heads = sorted({0, wl.Hv // 2 + 1, wl.Hv - 1})
    return streams, heads


def run_path(p, mode):
    if mode == "run":
        p.run()
    elif mode == "split":
        p.front_end()
        p.recurrence()
    elif mode == "seg":
        p.front_end()
        p.recurrence_segmented(2)
    else:
        raise ValueError(mode)


def check_workload(wl, cuda, pad_fill=0.0, seed=0, mode="run"):
    inp = make_inputs(wl, device=cuda, seed=seed)
    lengths = inp["lengths"]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    streams, heads = sample_units(wl, lengths)
    keep = {s: dict(x=inp["x"][cu[s]:cu[s + 1]].cpu(), conv_state=inp["conv_state"][s].cpu(),
                    h=inp["h"][s].cpu(), g=inp["g"][cu[s]:cu[s + 1]].cpu(),
                    beta=inp["beta"][cu[s]:cu[s + 1]].cpu()) for s in streams}
    conv_w = inp["conv_w"].cpu()
    p = PrefillPass(wl, inp, pad_fill=pad_fill)
    run_path(p, mode)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    act = wl.dtype
    d = wl.d
    worst_o, worst_h = 0.0, 0.0
    for s in streams:
        k_ = keep[s]
        L = lengths[s]
        q, k, v, new_conv = oracle_front(k_["x"], conv_w, k_["conv_state"][None], [L], wl.Hk,
                                         wl.Hv, d, 1e-6, act)
        np.testing.assert_array_equal(f64(inp["conv_state"][s].cpu()), new_conv[0])
        ref_o, ref_h = oracle_recurrence(k_["h"][None], q, k, v, k_["g"], k_["beta"], [L],
                                         1.0 / math.sqrt(d), wl.variant == "kda", heads=heads)
        got_o = f64(p.out[cu[s]:cu[s + 1]][:, heads].cpu())
        got_h = f64(inp["h"][s][heads].cpu())
        worst_o = max(worst_o, max_abs(got_o, ref_o))
        worst_h = max(worst_h, rel_frob(got_h, ref_h[0]))
    tol = TOL[act]
    print(f"\n[parity] {wl.name} ({mode}): max|o-o_ref| = {worst_o:.3e} (bar {tol['out']:.0e}), "
          f"state rel.Frobenius = {worst_h:.3e} (bar {tol['state']:.0e})")
    assert worst_o <= tol["out"], f"{wl.name}: max |o - o_ref| = {worst_o:.3g}"
    assert worst_h <= tol["state"], f"{wl.name}: state rel. Frobenius error {worst_h:.3g}"
    return p


def _paths():
    """(workload, path) pairs: every path PrefillPass offers for the workload."""
    for name, wl in WORKLOADS.items():
        tc = wl.dtype == "bf16" and wl.d == 128
        yield name, "run"
        if tc:  # run() is the one-launch path there; the two-launch path is a separate kernel
            yield name, "split"
        if tc and wl.B == 1:
            yield name, "seg"


@pytest.mark.parametrize("name,mode", list(_paths()))
def test_workload_full_size_sampled_parity(cuda, name, mode):
    check_workload(WORKLOADS[name], cuda, mode=mode)
    torch.cuda.empty_cache()


def test_kda_t4096_pad_fill_identical(cuda):
    """T = 4096 is a multiple of the chunk (no pad tail), so also run T = 4001."""
    for T in (4096, 4001):
        wl = WORKLOADS["kda_t4096_h32_d128"].replace(lengths=f"fixed:{T}")
        outs = []
        for pf in (0.0, 1e3):
            inp = make_inputs(wl, device="cuda", seed=1)
            p = PrefillPass(wl, inp, pad_fill=pf)
            p.run()
            torch.cuda.synchronize()
            outs.append((p.out.clone(), inp["h"].clone(), inp["conv_state"].clone()))
        for a, b in zip(*outs):
            assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["gdn_batched_8x2048_h16_d128", "kda_t4096_h32_d128"])
@pytest.mark.parametrize("mode", ["split", "fused"])
def test_graph_replay_equals_direct_calls(cuda, name, mode):
    """The bench also times each path as a CUDA-graph replay of the same public calls: two
    replayed steps must give the bits of two directly launched ones (outputs, h states, conv
    states), from the same inputs."""
    wl = WORKLOADS[name]
    res = []
    for graphed in (False, True):  # the direct run first: it also loads every kernel
        inp = make_inputs(wl, device=cuda, seed=3)
        p = PrefillPass(wl, inp)

        def body():
            if mode == "fused":
                p.fused()
            else:
                p.front_end()
                p.recurrence()
        if graphed:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                body()  # recorded, not run: the inputs are still the initial ones
            torch.cuda.synchronize()
            g.replay()
            g.replay()
        else:
            body()
            body()
        torch.cuda.synchronize()
        res.append((p.out.clone(), inp["h"].clone(), inp["conv_state"].clone()))
        del p, inp
    for a, b in zip(*res):
        assert torch.equal(a, b)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["kda_varlen_64_h32_d128", "gdn_varlen_32_hk16_hv32_d128",
                                  "gdn_batched_8x2048_h16_d128"])
def test_recurrence_repeatable_bitwise(cuda, name):
    """The recurrence run three times on the same inputs (h states restored in between) gives the
    same bits. The blocks claim their (stream, v-head) units from an atomic counter, so each run
    places the units on the SMs differently and the warps of a chunk meet with different skews: a
    hand-over between them that a barrier does not order would show as a difference."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, device=cuda, seed=5)
    p = PrefillPass(wl, inp)
    p.front_end()
    h0 = inp["h"].clone()
    res = []
    for _ in range(3):
        inp["h"].copy_(h0)
        p.recurrence()
        torch.cuda.synchronize()
        assert la.device_status() == 0
        res.append((p.out.clone(), inp["h"].clone()))
    for out, h in res[1:]:
        assert torch.equal(out, res[0][0])
        assert torch.equal(h, res[0][1])
    del p, inp, res
    torch.cuda.empty_cache()
