"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by element.

Sizes span several 64-token chunks and ragged tails; edge cases cover empty streams, streams
shorter than the conv window, single tokens, pad_fill invariance (0, 1e3, NaN), guard bands,
batched == per-stream, split calls with carried state, and bad cu_seqlens.
"""
import math

import numpy as np
import pytest
import torch

import linear_attention_chunked_conv1d_gb300 as la
from linear_attention_chunked_conv1d_gb300.inputs import recurrence_inputs
from tests.helpers import (TOL, act_name, bf16_ulp_diff, f64, max_abs, oracle_recurrence,
                           rel_frob)
import oracle

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def gen(seed):
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    return g


# ------------------------------------------------------------------------------------ conv
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("lengths", [[100], [1], [2, 0, 1, 70, 130, 3, 64, 65]])
# C = 100: fp32 rows of whole 16-byte vectors that are not whole warps of channel quads
@pytest.mark.parametrize("dtype,C", [("f32", 96), ("f32", 100), ("bf16", 96)])
def test_conv_parity(cuda, dtype, K, lengths, C):
    g = gen(K * 7 + len(lengths))
    T = sum(lengths)
    B = len(lengths)
    x = torch.randn(T, C + 32, generator=g).to(DT[dtype])      # row stride > channels
    w = (torch.randn(C, K, generator=g) * 0.25).to(DT[dtype])
    st = torch.randn(B, max(K - 1, 1), C, generator=g).to(DT[dtype])[:, :K - 1]
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)
    xd, wd, std = x.to(cuda), w.to(cuda), st.contiguous().to(cuda)
    out = torch.full((T + 8, C + 16), 7.0, dtype=DT[dtype], device=cuda)  # 8 guard rows
    if B == 1:
        la.conv1d_silu_prefill(std[0] if K > 1 else None, xd[:, :C], wd, out[:T, :C], t=T)
    else:
        ptrs = la.pointer_array([std[s] for s in range(B)]) if K > 1 else \
            torch.zeros(B, dtype=torch.int64, device=cuda)
        la.conv1d_silu_prefill_varlen(ptrs, xd[:, :C], wd, out[:T, :C], cu.to(cuda),
                                      total_tokens=T)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    ref_out, ref_st = oracle.conv1d_silu_varlen(f64(st), f64(x)[:, :C], f64(w), cu.numpy())
    got = out[:T, :C].cpu()
    if dtype == "f32":
        assert max_abs(f64(got), ref_out) <= 1e-5 * max(1.0, np.abs(ref_out).max())
    else:
        assert bf16_ulp_diff(got, ref_out) <= 1
    assert torch.all(out[T:].cpu() == 7.0) and torch.all(out[:T, C:].cpu() == 7.0)
    if K > 1:
        np.testing.assert_array_equal(f64(std.cpu()), ref_st)


def test_conv_split_call_carries_state(cuda):
    g = gen(3)
    C, K, T, cut = 64, 4, 150, 61
    x = torch.randn(T, C, generator=g).to(torch.bfloat16).to(cuda)
    w = (torch.randn(C, K, generator=g) * 0.25).to(torch.bfloat16).to(cuda)
    st0 = torch.randn(K - 1, C, generator=g).to(torch.bfloat16).to(cuda)
    a, b = st0.clone(), st0.clone()
    o1 = torch.empty_like(x)
    o2 = torch.empty_like(x)
    la.conv1d_silu_prefill(a, x, w, o1)
    la.conv1d_silu_prefill(b, x[:cut], w, o2[:cut])
    la.conv1d_silu_prefill(b, x[cut:], w, o2[cut:])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(a, b)


# ------------------------------------------------------------------------------------ L2
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hd", [64, 128])
def test_l2_parity(cuda, dtype, hd):
    g = gen(hd)
    t, H = 77, 6
    x = torch.randn(t, H * hd + 64, generator=g).to(DT[dtype])
    x[5, :hd] = 0
    xd = x.to(cuda)
    la.l2norm_heads(xd, H - 1, hd, eps=1e-6)
    torch.cuda.synchronize()
    ref = oracle.l2norm_heads(f64(x), H - 1, hd, 1e-6)
    got = xd.cpu()
    if dtype == "f32":
        assert max_abs(f64(got), ref) <= 1e-6
    else:
        assert bf16_ulp_diff(got, ref) <= 1
    assert torch.equal(got[:, (H - 1) * hd:], x[:, (H - 1) * hd:])  # last head untouched


# ------------------------------------------------------------------------------------ recurrence
def run_rec(cuda, inp, Hk, Hv, d, *, kda, mode, pad_fill=0.0, scale=None, guard=0):
    """Run one recurrence call on GPU; returns (out [T][Hv][d] cpu, states [B][Hv][d][d] cpu)."""
    lengths = inp["lengths"]
    T = sum(lengths)
    B = len(lengths)
    q, k, v = (inp[n].to(cuda) for n in ("q", "k", "v"))
    q, k, v = (a.reshape(T, -1) for a in (q, k, v))
    g, beta = inp["g"].to(cuda), inp["beta"].to(cuda)
    h = inp["h"].clone().to(cuda)
    out_full = torch.full((T + guard, Hv, d), 3.0, dtype=q.dtype, device=cuda)
    out = out_full[:T]
    ptrs = la.pointer_array([h[s] for s in range(B)])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    cu = inp["cu_seqlens"].to(cuda)
    nbytes = la.prefill_workspace_bytes(B, T, Hk, Hv, d, d, q.dtype)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=cuda) if nbytes else None
    if kda:
        la.kda_prefill(ptrs, q, k, v, g, beta, out, None if mode == "single" else cu,
                       Hk=Hk, Hv=Hv, dk=d, dv=d, max_seqlen=max(lengths), scale=scale,
                       pad_fill=pad_fill, workspace=ws)
    elif mode == "batched":
        la.gdn_prefill_batched(ptrs, q, k, v, g, beta, out, B=B, T=lengths[0], Hk=Hk, Hv=Hv,
                               dk=d, dv=d, scale=scale, workspace=ws)
    else:
        la.gdn_prefill_varlen(ptrs, q, k, v, g, beta, out, cu, max_seqlen=max(lengths), Hk=Hk,
                              Hv=Hv, dk=d, dv=d, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    if guard:
        assert torch.all(out_full[T:].cpu() == 3.0), "write past the last token"
    return out.cpu(), h.cpu()


def check_parity(inp, got_out, got_h, Hk, Hv, d, kda, dtype):
    scale = 1.0 / math.sqrt(d)
    ref_out, ref_h = oracle_recurrence(inp["h"], inp["q"], inp["k"], inp["v"], inp["g"],
                                       inp["beta"], inp["lengths"], scale, kda)
    tol = TOL[dtype]
    e_out = max_abs(f64(got_out), ref_out)
    e_h = rel_frob(f64(got_h), ref_h)
    print(f"\n[parity] {dtype} d={d} kda={kda}: max|o-o_ref| = {e_out:.3e}, "
          f"state rel.Frobenius = {e_h:.3e}")
    assert e_out <= tol["out"], f"max |o - o_ref| = {e_out:.3g} > {tol['out']}"
    assert e_h <= tol["state"], f"state rel. Frobenius error {e_h:.3g} > {tol['state']}"
    return e_out, e_h


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_gdn_batched_parity(cuda, dtype, d):
    inp = recurrence_inputs([150] * 3, 2, 2, d, dtype=dtype, seed=d)
    o, h = run_rec(cuda, inp, 2, 2, d, kda=False, mode="batched", guard=5)
    check_parity(inp, o, h, 2, 2, d, False, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_gdn_varlen_gqa_parity(cuda, dtype, d):
    lengths = [1, 64, 65, 200, 0, 37, 128]
    inp = recurrence_inputs(lengths, 2, 4, d, dtype=dtype, seed=11 + d)
    o, h = run_rec(cuda, inp, 2, 4, d, kda=False, mode="varlen", guard=3)
    check_parity(inp, o, h, 2, 4, d, False, dtype)
    # zero-length stream: state untouched
    assert torch.equal(h[4], inp["h"][4])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode", ["single", "varlen"])
def test_kda_parity(cuda, dtype, d, mode):
    lengths = [201] if mode == "single" else [130, 3, 64, 0, 99]
    inp = recurrence_inputs(lengths, 2, 2, d, kda=True, dtype=dtype, seed=5 + d)
    o, h = run_rec(cuda, inp, 2, 2, d, kda=True, mode=mode, guard=2)
    check_parity(inp, o, h, 2, 2, d, True, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kda_pad_fill_invariance_bitwise(cuda, dtype):
    inp = recurrence_inputs([100], 2, 2, 128, kda=True, dtype=dtype, seed=77)
    base = run_rec(cuda, inp, 2, 2, 128, kda=True, mode="single", pad_fill=0.0)
    for pf in (1e3, float("nan"), -7.5):
        o, h = run_rec(cuda, inp, 2, 2, 128, kda=True, mode="single", pad_fill=pf)
        assert torch.equal(o, base[0]) and torch.equal(h, base[1]), pf


def test_pad_rows_in_caller_buffers_ignored(cuda):
    """Rows of the caller's q/k/v/g/beta past t (garbage, 1e3, NaN) do not reach the results."""
    inp = recurrence_inputs([100], 2, 2, 128, kda=True, dtype="bf16", seed=78)
    base = run_rec(cuda, inp, 2, 2, 128, kda=True, mode="single")
    padded = dict(inp)
    for name, val in (("q", 1e3), ("k", float("nan")), ("v", 1e3), ("g", float("nan")),
                      ("beta", 1e3)):
        a = inp[name]
        tail = torch.full((28,) + tuple(a.shape[1:]), val, dtype=a.dtype)
        padded[name] = torch.cat([a, tail])
    # the same call over the first T tokens of the longer buffers
    T, d, Hk, Hv = 100, 128, 2, 2
    qd, kd, vd = (padded[n].to(cuda).reshape(padded[n].shape[0], -1) for n in ("q", "k", "v"))
    gd, bd = padded["g"].to(cuda), padded["beta"].to(cuda)
    h = inp["h"].clone().to(cuda)
    out = torch.empty(T, Hv, d, dtype=torch.bfloat16, device=cuda)
    ws = torch.empty(la.prefill_workspace_bytes(1, T, Hk, Hv, d, d, la.LA_BF16),
                     dtype=torch.uint8, device=cuda)
    la.kda_prefill(la.pointer_array([h[0]]), qd, kd, vd, gd, bd, out, None, Hk=Hk, Hv=Hv, dk=d,
                   dv=d, total_tokens=T, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), base[0]) and torch.equal(h.cpu(), base[1])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_batched_equals_varlen_and_per_stream_bitwise(cuda, dtype):
    lengths = [130] * 3
    inp = recurrence_inputs(lengths, 2, 4, 128, dtype=dtype, seed=21)
    ob, hb = run_rec(cuda, inp, 2, 4, 128, kda=False, mode="batched")
    ov, hv = run_rec(cuda, inp, 2, 4, 128, kda=False, mode="varlen")
    assert torch.equal(ob, ov) and torch.equal(hb, hv)
    for s in range(3):
        sl = slice(130 * s, 130 * (s + 1))
        one = {n: inp[n][sl] for n in ("q", "k", "v", "g", "beta")}
        one.update(h=inp["h"][s:s + 1], lengths=[130],
                   cu_seqlens=torch.tensor([0, 130], dtype=torch.int32))
        o1, h1 = run_rec(cuda, one, 2, 4, 128, kda=False, mode="batched")
        assert torch.equal(o1, ob[sl]) and torch.equal(h1[0], hb[s])


@pytest.mark.parametrize("kda", [False, True])
def test_split_call_with_carried_state(cuda, kda):
    T, cut = 300, 97
    inp = recurrence_inputs([T], 2, 2, 128, kda=kda, dtype="bf16", seed=31)
    o_all, h_all = run_rec(cuda, inp, 2, 2, 128, kda=kda, mode="single" if kda else "varlen")
    a = {n: inp[n][:cut] for n in ("q", "k", "v", "g", "beta")}
    a.update(h=inp["h"], lengths=[cut], cu_seqlens=torch.tensor([0, cut], dtype=torch.int32))
    oa, ha = run_rec(cuda, a, 2, 2, 128, kda=kda, mode="single" if kda else "varlen")
    b = {n: inp[n][cut:] for n in ("q", "k", "v", "g", "beta")}
    b.update(h=ha, lengths=[T - cut], cu_seqlens=torch.tensor([0, T - cut], dtype=torch.int32))
    ob, hb = run_rec(cuda, b, 2, 2, 128, kda=kda, mode="single" if kda else "varlen")
    assert max_abs(f64(torch.cat([oa, ob])), f64(o_all)) <= 2e-3
    assert rel_frob(f64(hb), f64(h_all)) <= 1e-3
    # and the split result is itself within the bar of the oracle
    check_parity(inp, torch.cat([oa, ob]), hb, 2, 2, 128, kda, "bf16")


def test_bad_cu_seqlens_raise_device_status(cuda):
    inp = recurrence_inputs([50, 50], 1, 1, 64, dtype="bf16", seed=41)
    T = 100
    q, k, v = (inp[n].to(cuda).reshape(T, -1) for n in ("q", "k", "v"))
    h = inp["h"].clone().to(cuda)
    out = torch.zeros(T, 1, 64, dtype=torch.bfloat16, device=cuda)
    bad = torch.tensor([0, 70, 60], dtype=torch.int32, device=cuda)  # decreasing
    la.device_status()
    la.gdn_prefill_varlen(la.pointer_array([h[0], h[1]]), q, k, v, inp["g"].to(cuda),
                          inp["beta"].to(cuda), out, bad, max_seqlen=70, Hk=1, Hv=1, dk=64,
                          dv=64, total_tokens=T)
    assert la.device_status() & la.LA_DEV_BAD_SEQLENS
    assert la.device_status() == 0  # cleared


def test_refusal_leaves_buffers_untouched(cuda):
    inp = recurrence_inputs([64], 1, 1, 64, dtype="bf16", seed=42)
    q, k, v = (inp[n].to(cuda).reshape(64, -1) for n in ("q", "k", "v"))
    h = inp["h"].clone().to(cuda)
    out = torch.full((64, 1, 64), 5.0, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(la.LinAttnError) as ei:
        la.gdn_prefill_batched(la.pointer_array([h[0]]), q, k, v, inp["g"].to(cuda),
                               inp["beta"].to(cuda), out, B=1, T=64, Hk=1, Hv=1, dk=64, dv=64,
                               max_tokens=63)
    assert ei.value.code == la.LA_ERR_COUNT
    torch.cuda.synchronize()
    assert torch.all(out.cpu() == 5.0) and torch.equal(h.cpu(), inp["h"])


def test_kda_extreme_gates_exact_path(cuda):
    """Half-chunk decays beyond e^80 in some channels: the tensor-core kernel must take its exact
    pairwise-exponent path for those chunks and still match the oracle."""
    inp = recurrence_inputs([150], 2, 2, 128, kda=True, dtype="bf16", seed=91)
    g = inp["g"].clone()
    g[:, :, :8] = -12.0          # 8 channels decay by e^-12 per token
    g[40:60, 1, 100:] = -30.0    # and a burst on another head
    inp["g"] = g
    o, h = run_rec(cuda, inp, 2, 2, 128, kda=True, mode="single")
    assert torch.isfinite(o.float()).all() and torch.isfinite(h).all()
    check_parity(inp, o, h, 2, 2, 128, True, "bf16")


def test_bad_cu_seqlens_tensor_core_path(cuda):
    inp = recurrence_inputs([50, 50], 1, 1, 128, dtype="bf16", seed=43)
    T = 100
    q, k, v = (inp[n].to(cuda).reshape(T, -1) for n in ("q", "k", "v"))
    h = inp["h"].clone().to(cuda)
    out = torch.zeros(T, 1, 128, dtype=torch.bfloat16, device=cuda)
    ws = torch.empty(la.prefill_workspace_bytes(2, T, 1, 1, 128, 128, la.LA_BF16),
                     dtype=torch.uint8, device=cuda)
    bad = torch.tensor([0, 70, 60], dtype=torch.int32, device=cuda)
    la.device_status()
    la.gdn_prefill_varlen(la.pointer_array([h[0], h[1]]), q, k, v, inp["g"].to(cuda),
                          inp["beta"].to(cuda), out, bad, max_seqlen=70, Hk=1, Hv=1, dk=128,
                          dv=128, total_tokens=T, workspace=ws)
    assert la.device_status() & la.LA_DEV_BAD_SEQLENS


def test_workspace_too_small_is_refused(cuda):
    inp = recurrence_inputs([64], 1, 1, 128, dtype="bf16", seed=44)
    q, k, v = (inp[n].to(cuda).reshape(64, -1) for n in ("q", "k", "v"))
    h = inp["h"].clone().to(cuda)
    out = torch.zeros(64, 1, 128, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(la.LinAttnError) as ei:
        la.gdn_prefill_batched(la.pointer_array([h[0]]), q, k, v, inp["g"].to(cuda),
                               inp["beta"].to(cuda), out, B=1, T=64, Hk=1, Hv=1, dk=128, dv=128)
    assert ei.value.code == la.LA_ERR_ARG


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("lengths", [[150], [1, 0, 70, 3, 129, 64]])
def test_fused_conv_l2_equals_two_launches_and_oracle(cuda, dtype, hd, lengths):
    g = gen(hd + len(lengths))
    Hk, Hv, K = 2, 3, 4
    C = 2 * Hk * hd + Hv * hd
    T, B = sum(lengths), len(lengths)
    x = torch.randn(T, C, generator=g).to(DT[dtype])
    w = (torch.randn(C, K, generator=g) * 0.25).to(DT[dtype])
    st = torch.randn(B, K - 1, C, generator=g).to(DT[dtype])
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)
    xd, wd, cud = x.to(cuda), w.to(cuda), cu.to(cuda)
    st1, st2 = st.clone().to(cuda), st.clone().to(cuda)
    o1 = torch.empty(T, C, dtype=DT[dtype], device=cuda)
    o2 = torch.full((T, C), 9.0, dtype=DT[dtype], device=cuda)
    p1 = la.pointer_array([st1[s] for s in range(B)])
    p2 = la.pointer_array([st2[s] for s in range(B)])
    if B == 1:
        la.conv1d_silu_prefill(st1[0], xd, wd, o1)
    else:
        la.conv1d_silu_prefill_varlen(p1, xd, wd, o1, cud)
    la.l2norm_heads(o1, 2 * Hk, hd, eps=1e-6)
    la.conv1d_silu_l2_prefill(p2, xd, wd, o2, None if B == 1 else cud, l2_heads=2 * Hk,
                              head_dim=hd, eps=1e-6)
    torch.cuda.synchronize()
    assert la.device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(st1, st2)
    q, k, v, ref_st = oracle.front_end(f64(x), f64(w), f64(st), cu.numpy(), Hk=Hk, Hv=Hv,
                                       dk=hd, dv=hd, eps=1e-6, act_dtype=dtype)
    ref = np.concatenate([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], axis=1)
    got = o2.cpu()
    if dtype == "f32":
        assert max_abs(f64(got), ref) <= 1e-5
    else:
        assert bf16_ulp_diff(got, ref) <= 1
    np.testing.assert_array_equal(f64(st2.cpu()), ref_st)


def test_gdn_extreme_gates_exact_decay_path(cuda):
    """Half-chunk decays beyond e^80 (g = -12 per token): the tensor-core kernel must use the
    exact pairwise decay instead of the row x column factorisation, and still match."""
    inp = recurrence_inputs([200, 77], 2, 4, 128, dtype="bf16", seed=93)
    g = inp["g"].clone()
    g[:, 1] = -12.0
    g[60:140, 2] = -30.0
    inp["g"] = g
    o, h = run_rec(cuda, inp, 2, 4, 128, kda=False, mode="varlen")
    assert torch.isfinite(o.float()).all() and torch.isfinite(h).all()
    check_parity(inp, o, h, 2, 4, 128, False, "bf16")


def test_kda_decay_near_split_limit(cuda):
    """KDA's D1 splits each decay as e^{gc_t} e^{-gc_i}; the fast path holds while a chunk's
    decay stays below e^80 in every channel. Channels decaying by e^-78 per chunk (just inside)
    and by e^-83 (just past, exact path) must both match the oracle."""
    inp = recurrence_inputs([64 * 4, 100], 1, 2, 128, kda=True, dtype="bf16", seed=95)
    g = inp["g"].clone()
    g[:, 0, :16] = -78.0 / 64    # fast path at its edge: e^{-gc} up to e^78
    g[:, 1, 16:24] = -83.0 / 64  # the exact pairwise path
    inp["g"] = g
    o, h = run_rec(cuda, inp, 1, 2, 128, kda=True, mode="varlen")
    assert torch.isfinite(o.float()).all() and torch.isfinite(h).all()
    check_parity(inp, o, h, 1, 2, 128, True, "bf16")


@pytest.mark.parametrize("kda", [False, True])
def test_next_stream_rows_do_not_reach_a_stream(cuda, kda):
    """The tensor-core path loads 64-row boxes, so a stream's last chunk also brings rows of the
    next stream; they are rewritten (pad value, zero V) before any use. A stream's outputs and
    state must keep their bits whatever the next stream holds, NaN included."""
    lengths = [70, 50]
    inp = recurrence_inputs(lengths, 1, 2, 128, kda=kda, dtype="bf16", seed=97)
    o_a, h_a = run_rec(cuda, inp, 1, 2, 128, kda=kda, mode="varlen")
    poisoned = dict(inp)
    for name in ("q", "k", "v"):
        t = inp[name].clone()
        t[lengths[0]:] = float("nan")
        poisoned[name] = t
    o_b, h_b = run_rec(cuda, poisoned, 1, 2, 128, kda=kda, mode="varlen")
    assert torch.equal(o_a[:lengths[0]], o_b[:lengths[0]])
    assert torch.equal(h_a[0], h_b[0])
    check_parity(inp, o_a, h_a, 1, 2, 128, kda, "bf16")
