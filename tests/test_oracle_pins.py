"""Pins of the fp64 oracle against things other than itself (CPU only).

- a hand-worked example (tests/golden/gated_delta_hand.json, exact decimals derived by hand);
- brute force: S_T = S_0 M_1..M_T + sum_t beta_t v_t k_t^T M_{t+1}..M_T with
  M_t = diag(alpha_t)(I - beta_t k_t k_t^T), as explicit dense matrix products;
- closed forms and special cases of the gated delta rule;
- conv1d against numpy.convolve and scipy's logistic function; L2 norm against numpy.linalg;
- invariants: batched == per stream, split call with carried state == one call, GQA mapping,
  thread-count independence, and the chunked (WY) restatement == token by token.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
from tests.chunk_algebra import chunked_unit

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gated_delta_hand.json")


def rng(seed):
    return np.random.default_rng(seed)


def rand_unit_inputs(r, T, dk, dv, per_channel, Hk=1, Hv=1):
    q = r.standard_normal((T, Hk, dk)) / np.sqrt(dk)
    k = r.standard_normal((T, Hk, dk)) / np.sqrt(dk)
    v = r.standard_normal((T, Hv, dv)) * 0.5
    g = -np.log1p(np.exp(r.standard_normal((T, Hv, dk) if per_channel else (T, Hv))))
    beta = expit(r.standard_normal((T, Hv)))
    return q, k, v, g, beta


def run_oracle(h, q, k, v, g, beta, lengths, scale, per_channel, threads=None):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return oracle.gated_delta(h, q, k, v, g, beta, cu, scale=scale, per_channel=per_channel,
                              threads=threads)


# ---------------------------------------------------------------- hand-worked golden example
@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_golden_hand_example(variant):
    G = json.load(open(GOLDEN))[variant]
    S0 = np.array(G["S0"], dtype=float)
    k = np.array(G["k"], dtype=float)[:, None, :]
    q = np.array(G["q"], dtype=float)[:, None, :]
    v = np.array(G["v"], dtype=float)[:, None, :]
    T = k.shape[0]
    g = np.array(G["g"], dtype=float).reshape(T, 1, -1) if variant == "kda" else \
        np.array(G["g"], dtype=float).reshape(T, 1)
    beta = np.array(G["beta"], dtype=float).reshape(T, 1)
    h = S0.T[None, None]  # H = S^T, [B][Hv][dk][dv]
    out, h1 = run_oracle(h, q, k, v, g, beta, [T], 1.0, variant == "kda")
    np.testing.assert_allclose(out[:, 0, :], np.array(G["o"]), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(h1[0, 0].T, np.array(G["S_final"]), rtol=1e-13, atol=1e-13)


def test_golden_hand_conv():
    G = json.load(open(GOLDEN))["conv"]
    out, st = oracle.conv1d_silu(np.array(G["state"]), np.array(G["x"]), np.array(G["w"]))
    y = np.array(G["y_pre_silu"], dtype=float)
    np.testing.assert_allclose(out, y * expit(y), rtol=1e-15)
    np.testing.assert_array_equal(st, np.array(G["new_state"]))


# ---------------------------------------------------------------- brute force
def brute_unit(S0, q, k, v, g, beta, scale):
    """Outputs and final S of one unit from explicit products of transition matrices."""
    T, dk = k.shape
    I = np.eye(dk)

    def M(t):
        a = np.exp(g[t]) * np.ones(dk)
        return np.diag(a) @ (I - beta[t] * np.outer(k[t], k[t]))

    outs = []
    for t in range(T):
        prod = I.copy()
        for s in range(t + 1):
            prod = prod @ M(s)
        St = S0 @ prod
        for s in range(t + 1):
            tail = I.copy()
            for r_ in range(s + 1, t + 1):
                tail = tail @ M(r_)
            St = St + beta[s] * np.outer(v[s], k[s]) @ tail
        outs.append(scale * St @ q[t])
    return np.array(outs), St


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("T,dk,dv", [(1, 2, 3), (5, 4, 4), (6, 3, 2)])
def test_brute_force_products(per_channel, T, dk, dv):
    r = rng(T * 100 + dk * 10 + dv + per_channel)
    q, k, v, g, beta = rand_unit_inputs(r, T, dk, dv, per_channel)
    S0 = r.standard_normal((dv, dk)) * 0.3
    out, h1 = run_oracle(S0.T[None, None], q, k, v, g, beta, [T], 0.7, per_channel)
    gg = g[:, 0] if per_channel else g[:, 0]
    ob, Sb = brute_unit(S0, q[:, 0], k[:, 0], v[:, 0], gg, beta[:, 0], 0.7)
    np.testing.assert_allclose(out[:, 0], ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h1[0, 0].T, Sb, rtol=1e-12, atol=1e-12)


def test_brute_force_gqa_multistream():
    """Two streams, Hk=1 shared by Hv=2 v-heads: each (stream, v-head) equals its brute force."""
    r = rng(7)
    lengths = [3, 4]
    T = sum(lengths)
    q, k, v, g, beta = rand_unit_inputs(r, T, 3, 2, True, Hk=1, Hv=2)
    S0 = r.standard_normal((2, 2, 2, 3)) * 0.3  # [B][Hv][dv][dk]
    out, h1 = run_oracle(np.transpose(S0, (0, 1, 3, 2)), q, k, v, g, beta, lengths, 1.0, True)
    off = 0
    for s, L in enumerate(lengths):
        sl = slice(off, off + L)
        for j in range(2):
            ob, Sb = brute_unit(S0[s, j], q[sl, 0], k[sl, 0], v[sl, j], g[sl, j], beta[sl, j], 1.0)
            np.testing.assert_allclose(out[sl, j], ob, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(h1[s, j].T, Sb, rtol=1e-12, atol=1e-12)
        off += L


# ---------------------------------------------------------------- closed forms
def test_beta_zero_pure_decay():
    r = rng(1)
    T, d = 7, 4
    q, k, v, g, beta = rand_unit_inputs(r, T, d, d, True)
    beta[:] = 0.0
    S0 = r.standard_normal((d, d))
    out, h1 = run_oracle(S0.T[None, None], q, k, v, g, beta, [T], 0.5, True)
    cum = np.cumsum(g[:, 0, :], axis=0)
    for t in range(T):
        np.testing.assert_allclose(out[t, 0], 0.5 * S0 @ (np.exp(cum[t]) * q[t, 0]), rtol=1e-13)
    np.testing.assert_allclose(h1[0, 0].T, S0 * np.exp(cum[-1])[None, :], rtol=1e-13)


def test_delta_write_is_exact():
    """beta = 1 and |k| = 1: after each step S_t k_t = v_t (read with q = k, scale 1)."""
    r = rng(2)
    T, d = 9, 5
    k = r.standard_normal((T, 1, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, 1, d))
    g = -np.abs(r.standard_normal((T, 1)))
    beta = np.ones((T, 1))
    out, _ = run_oracle(r.standard_normal((1, 1, d, d)), k, k, v, g, beta, [T], 1.0, False)
    np.testing.assert_allclose(out[:, 0], v[:, 0], rtol=1e-12, atol=1e-12)


def test_single_token_from_zero_state():
    r = rng(3)
    d = 6
    q, k, v, g, beta = rand_unit_inputs(r, 1, d, d, False)
    out, _ = run_oracle(np.zeros((1, 1, d, d)), q, k, v, g, beta, [1], 0.25, False)
    expect = 0.25 * beta[0, 0] * (k[0, 0] @ q[0, 0]) * v[0, 0]
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-14, atol=1e-16)


def test_orthonormal_keys_no_decay():
    """alpha = 1, beta = 1, orthonormal keys: S_T = S_0 (I - sum k k^T) + sum v k^T."""
    r = rng(4)
    d, T = 6, 4
    Qm, _ = np.linalg.qr(r.standard_normal((d, d)))
    k = Qm[:, :T].T[:, None, :]
    v = r.standard_normal((T, 1, d))
    S0 = r.standard_normal((d, d))
    _, h1 = run_oracle(S0.T[None, None], k, k, v, np.zeros((T, 1)), np.ones((T, 1)), [T], 1.0,
                       False)
    kk = sum(np.outer(k[t, 0], k[t, 0]) for t in range(T))
    vk = sum(np.outer(v[t, 0], k[t, 0]) for t in range(T))
    np.testing.assert_allclose(h1[0, 0].T, S0 @ (np.eye(d) - kk) + vk, rtol=1e-12, atol=1e-12)


def test_kda_with_broadcast_gate_equals_gdn():
    r = rng(5)
    T, d = 11, 4
    q, k, v, g, beta = rand_unit_inputs(r, T, d, d, False)
    h0 = r.standard_normal((1, 1, d, d))
    o1, h1 = run_oracle(h0, q, k, v, g, beta, [T], 0.3, False)
    o2, h2 = run_oracle(h0, q, k, v, np.repeat(g[:, :, None], d, axis=2), beta, [T], 0.3, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(h1, h2)


# ---------------------------------------------------------------- conv and L2
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("t", [1, 2, 5, 17])
def test_conv_matches_numpy_convolve(K, t):
    r = rng(K * 31 + t)
    C = 5
    state = r.standard_normal((K - 1, C))
    x = r.standard_normal((t, C))
    w = r.standard_normal((C, K))
    b = r.standard_normal(C)
    out, st = oracle.conv1d_silu(state, x, w, b)
    xh = np.concatenate([state, x], axis=0)
    for c in range(C):
        y = np.convolve(xh[:, c], w[c, ::-1], mode="valid") + b[c]
        np.testing.assert_allclose(out[:, c], y * expit(y), rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(st, xh[t:t + K - 1])


def test_conv_special_taps():
    r = rng(9)
    x = r.standard_normal((6, 3))
    w1 = r.standard_normal((3, 1))
    out, _ = oracle.conv1d_silu(np.zeros((0, 3)), x, w1)
    y = x * w1[:, 0]
    np.testing.assert_allclose(out, y * expit(y), rtol=1e-14)
    w = np.zeros((3, 4))
    w[:, 3] = 1.0  # e_{K-1}: the current token only
    out, _ = oracle.conv1d_silu(r.standard_normal((3, 3)), x, w)
    np.testing.assert_allclose(out, x * expit(x), rtol=1e-14)


def test_conv_varlen_short_streams_carry_state():
    """Streams shorter than kernel-1 keep part of the old state, in order."""
    r = rng(10)
    C, K = 2, 4
    lengths = [1, 0, 2, 5]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    x = r.standard_normal((cu[-1], C))
    states = r.standard_normal((len(lengths), K - 1, C))
    w = r.standard_normal((C, K))
    out, ns = oracle.conv1d_silu_varlen(states, x, w, cu)
    assert out.shape == x.shape
    for s, L in enumerate(lengths):
        xh = np.concatenate([states[s], x[cu[s]:cu[s + 1]]])
        np.testing.assert_array_equal(ns[s], xh[L:L + K - 1])
        # each stream's rows of the packed output are that stream's own single-stream conv,
        # which numpy.convolve over [its state ; its rows] gives independently
        own, _ = oracle.conv1d_silu(states[s], x[cu[s]:cu[s + 1]], w)
        np.testing.assert_array_equal(out[cu[s]:cu[s + 1]], own)
        if L == 0:
            continue
        for c in range(C):
            y = np.convolve(xh[:, c], w[c, ::-1], mode="valid")
            np.testing.assert_allclose(out[cu[s]:cu[s + 1], c], y * expit(y), rtol=1e-13,
                                       atol=1e-15)


def test_l2norm_properties():
    r = rng(11)
    t, H, d = 5, 3, 8
    x = r.standard_normal((t, H * d + 4))
    x[2, d:2 * d] = 0.0
    eps = 1e-6
    y = oracle.l2norm_heads(x, H, d, eps)
    for h in range(H):
        xs, ys = x[:, h * d:(h + 1) * d], y[:, h * d:(h + 1) * d]
        nx = np.linalg.norm(xs, axis=1)
        np.testing.assert_allclose(np.linalg.norm(ys, axis=1), nx / np.sqrt(nx ** 2 + eps),
                                   rtol=1e-14)
        nz = nx > 0
        np.testing.assert_allclose(ys[nz] * nx[nz, None], xs[nz] * np.linalg.norm(ys[nz], axis=1)[:, None],
                                   rtol=1e-13, atol=1e-15)
    assert np.all(y[2, d:2 * d] == 0.0)
    np.testing.assert_array_equal(y[:, H * d:], x[:, H * d:])  # channels past the heads untouched


# ---------------------------------------------------------------- the front end composition
def _bf16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).to(torch.float64).numpy()


def _front_by_hand(x, w, states, cu, Hk, Hv, d, eps, *, swap_qk=False, round_conv=True,
                   round_l2=True):
    """The front end rebuilt from library routines only: numpy.convolve per channel over
    [carried state ; the stream's rows] (reversed taps, valid mode), SiLU from scipy's logistic
    function, bf16 rounding by torch, the L2 norm of each q and k head row by numpy.linalg, and
    the [q heads | k heads | v heads] slices of the packed channels."""
    T, C = x.shape
    conv = np.zeros((T, C))
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        xh = np.concatenate([states[s], x[a:b]])
        for c in range(C):
            y = np.convolve(xh[:, c], w[c, ::-1], mode="valid")
            conv[a:b, c] = y * expit(y)
    if round_conv:
        conv = _bf16(conv)
    normed = conv.copy()
    for h in range(2 * Hk):
        blk = conv[:, h * d:(h + 1) * d]
        normed[:, h * d:(h + 1) * d] = blk / np.sqrt(np.sum(blk * blk, axis=1, keepdims=True) + eps)
    if round_l2:
        normed = _bf16(normed)
    q = normed[:, :Hk * d].reshape(T, Hk, d)
    k = normed[:, Hk * d:2 * Hk * d].reshape(T, Hk, d)
    v = normed[:, 2 * Hk * d:].reshape(T, Hv, d)
    return (k, q, v) if swap_qk else (q, k, v)


def test_front_end_composition_pinned():
    """oracle.front_end (conv -> bf16 -> L2 of the q|k heads -> bf16 -> [q | k | v] slices, the
    order of the conv_prefill, l2 and split launches of "glm5next_kda/prefill.rs") equals the
    same steps rebuilt from numpy/scipy/torch routines, on two streams with carried states, and
    the comparison is sensitive to a q/k swap and to a dropped rounding."""
    r = rng(21)
    Hk, Hv, d, K, eps = 1, 2, 4, 3, 1e-6
    lengths = [5, 3]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    cd = 2 * Hk * d + Hv * d
    x = _bf16(r.standard_normal((cu[-1], cd)))
    w = _bf16(r.standard_normal((cd, K)) * 0.5)
    states = _bf16(r.standard_normal((len(lengths), K - 1, cd)))
    q, k, v, ns = oracle.front_end(x, w, states, cu, Hk=Hk, Hv=Hv, dk=d, dv=d, eps=eps,
                                   act_dtype="bf16")
    eq, ek, ev = _front_by_hand(x, w, states, cu, Hk, Hv, d, eps)
    np.testing.assert_array_equal(q, eq)
    np.testing.assert_array_equal(k, ek)
    np.testing.assert_array_equal(v, ev)
    for s, L in enumerate(lengths):
        xh = np.concatenate([states[s], x[cu[s]:cu[s + 1]]])
        np.testing.assert_array_equal(ns[s], xh[L:L + K - 1])
    # q and k rows are unit vectors up to eps and bf16 rounding; v rows are not normalised
    assert np.allclose(np.linalg.norm(q, axis=2), 1.0, atol=1e-2)
    assert not np.allclose(np.linalg.norm(v, axis=2), 1.0, atol=1e-2)
    # planted mistakes: each one changes the result
    sq, sk, _ = _front_by_hand(x, w, states, cu, Hk, Hv, d, eps, swap_qk=True)
    assert not np.array_equal(sq, q) and not np.array_equal(sk, k)
    for kw in (dict(round_conv=False), dict(round_l2=False)):
        mq, mk, mv = _front_by_hand(x, w, states, cu, Hk, Hv, d, eps, **kw)
        assert not (np.array_equal(mq, q) and np.array_equal(mk, k) and np.array_equal(mv, v))


def test_front_end_fp32_keeps_fp32_rounding():
    """With fp32 activations the two stored steps round to fp32 (not bf16)."""
    r = rng(22)
    Hk, Hv, d, K, eps = 1, 1, 4, 4, 1e-6
    cu = np.array([0, 6])
    cd = 3 * d
    x = r.standard_normal((6, cd)).astype(np.float32).astype(np.float64)
    w = (r.standard_normal((cd, K)) * 0.5).astype(np.float32).astype(np.float64)
    st = np.zeros((1, K - 1, cd))
    q, k, v, _ = oracle.front_end(x, w, st, cu, Hk=Hk, Hv=Hv, dk=d, dv=d, eps=eps,
                                  act_dtype="f32")
    conv = np.zeros((6, cd))
    xh = np.concatenate([st[0], x])
    for c in range(cd):
        y = np.convolve(xh[:, c], w[c, ::-1], mode="valid")
        conv[:, c] = y * expit(y)
    conv = conv.astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(v.reshape(6, d), conv[:, 2 * d:])
    blk = conv[:, d:2 * d]
    ek = (blk / np.sqrt(np.sum(blk * blk, axis=1, keepdims=True) + eps)).astype(np.float32)
    np.testing.assert_array_equal(k.reshape(6, d), ek.astype(np.float64))


# ---------------------------------------------------------------- invariants
def test_batched_equals_per_stream_bitwise():
    r = rng(12)
    lengths = [5, 9, 1, 7]
    T = sum(lengths)
    q, k, v, g, beta = rand_unit_inputs(r, T, 4, 3, True, Hk=2, Hv=4)
    h0 = r.standard_normal((4, 4, 4, 3))
    out, h1 = run_oracle(h0, q, k, v, g, beta, lengths, 0.5, True)
    off = 0
    for s, L in enumerate(lengths):
        sl = slice(off, off + L)
        o_s, h_s = run_oracle(h0[s:s + 1], q[sl], k[sl], v[sl], g[sl], beta[sl], [L], 0.5, True)
        np.testing.assert_array_equal(out[sl], o_s)
        np.testing.assert_array_equal(h1[s], h_s[0])
        off += L


def test_split_call_equals_single_call_bitwise():
    r = rng(13)
    T, cut = 23, 10
    q, k, v, g, beta = rand_unit_inputs(r, T, 4, 4, False, Hk=1, Hv=2)
    h0 = r.standard_normal((1, 2, 4, 4))
    o_all, h_all = run_oracle(h0, q, k, v, g, beta, [T], 0.5, False)
    a, b = slice(0, cut), slice(cut, T)
    o_a, h_a = run_oracle(h0, q[a], k[a], v[a], g[a], beta[a], [cut], 0.5, False)
    o_b, h_b = run_oracle(h_a, q[b], k[b], v[b], g[b], beta[b], [T - cut], 0.5, False)
    np.testing.assert_array_equal(o_all, np.concatenate([o_a, o_b]))
    np.testing.assert_array_equal(h_all, h_b)
    # conv state carried across the split as well
    x = r.standard_normal((T, 6))
    w = r.standard_normal((6, 4))
    st0 = r.standard_normal((3, 6))
    out_all, st_all = oracle.conv1d_silu(st0, x, w)
    out_a, st_a = oracle.conv1d_silu(st0, x[:cut], w)
    out_b, st_b = oracle.conv1d_silu(st_a, x[cut:], w)
    np.testing.assert_array_equal(out_all, np.concatenate([out_a, out_b]))
    np.testing.assert_array_equal(st_all, st_b)


def test_thread_count_independent():
    r = rng(14)
    lengths = [13, 4, 20]
    q, k, v, g, beta = rand_unit_inputs(r, sum(lengths), 4, 4, True, Hk=1, Hv=3)
    h0 = r.standard_normal((3, 3, 4, 4))
    o1, h1 = run_oracle(h0, q, k, v, g, beta, lengths, 0.5, True, threads=1)
    o2, h2 = run_oracle(h0, q, k, v, g, beta, lengths, 0.5, True, threads=5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(h1, h2)


def test_zero_length_stream_is_noop():
    r = rng(15)
    lengths = [3, 0, 2]
    q, k, v, g, beta = rand_unit_inputs(r, 5, 4, 4, False)
    h0 = r.standard_normal((3, 1, 4, 4))
    _, h1 = run_oracle(h0, q, k, v, g, beta, lengths, 1.0, False)
    np.testing.assert_array_equal(h1[1], h0[1])


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("T,C", [(1, 64), (63, 64), (64, 64), (150, 64), (37, 8), (100, 16)])
def test_chunked_restatement_equals_token_by_token(per_channel, T, C):
    r = rng(T + C + per_channel)
    d = 8
    q, k, v, g, beta = rand_unit_inputs(r, T, d, d, per_channel)
    h0 = r.standard_normal((1, 1, d, d)) * 0.1
    out, h1 = run_oracle(h0, q, k, v, g, beta, [T], 0.4, per_channel)
    oc, hc = chunked_unit(h0[0, 0], q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0],
                          scale=0.4, C=C)
    np.testing.assert_allclose(oc, out[:, 0], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(hc, h1[0, 0], rtol=1e-10, atol=1e-10)


def test_planted_mistake_is_caught():
    """A dropped decay (alpha forced to 1) in the oracle's input is visible to the brute force."""
    r = rng(16)
    q, k, v, g, beta = rand_unit_inputs(r, 4, 3, 3, False)
    S0 = r.standard_normal((3, 3))
    out, _ = run_oracle(S0.T[None, None], q, k, v, np.zeros_like(g), beta, [4], 1.0, False)
    ob, _ = brute_unit(S0, q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], 1.0)
    assert np.max(np.abs(out[:, 0] - ob)) > 1e-3


# ---------------------------------------------------------------- gated RMSNorm (phase-3 epilogue)
def test_gated_rmsnorm_constant_row_closed_form():
    """o = 3 on every channel, eps = 7: 3 / sqrt(9 + 7) = 3/4; SiLU(ln 3) = (3/4) ln 3 since
    sigmoid(ln 3) = 3/4; with w = 2 every output is 2 (3/4)(3/4) ln 3."""
    dv = 16
    o = np.full((2, 3, dv), 3.0)
    z = np.full_like(o, math.log(3.0))
    y = oracle.gated_rmsnorm(o, z, np.full(dv, 2.0), 7.0)
    np.testing.assert_allclose(y, 2 * 0.75 * 0.75 * math.log(3.0), rtol=1e-14)
    y = oracle.gated_rmsnorm(-o, z, np.full(dv, 2.0), 7.0)  # odd in o
    np.testing.assert_allclose(y, -2 * 0.75 * 0.75 * math.log(3.0), rtol=1e-14)


def test_gated_rmsnorm_unit_rms_and_scale_invariance():
    """eps = 0, w = 1, z = 60 (SiLU(60) = 60 to double precision): y / 60 has RMS exactly 1
    over each row, and scaling o by c > 0 leaves y unchanged."""
    r = rng(21)
    dv = 128
    o = r.standard_normal((5, 4, dv))
    z = np.full_like(o, 60.0)
    y = oracle.gated_rmsnorm(o, z, np.ones(dv), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean((y / 60.0) ** 2, axis=-1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.gated_rmsnorm(37.5 * o, z, np.ones(dv), 0.0), y,
                               rtol=1e-13)


def test_gated_rmsnorm_gate_limits_and_channel_weights():
    """SiLU(0) = 0 and SiLU(-800) = -0: those outputs vanish; the weight scales its own channel
    only (a transposed or shared weight would not)."""
    r = rng(22)
    dv = 64
    o = r.standard_normal((3, 2, dv))
    z = r.standard_normal((3, 2, dv))
    z[0, 0, :] = 0.0
    z[1, 1, :] = -800.0
    w = r.uniform(0.5, 2.0, dv)
    y1 = oracle.gated_rmsnorm(o, z, np.ones(dv), 1e-6)
    yw = oracle.gated_rmsnorm(o, z, w, 1e-6)
    assert np.all(y1[0, 0] == 0.0) and np.all(y1[1, 1] == 0.0)
    mask = y1 != 0
    np.testing.assert_allclose((yw[mask] / y1[mask]), np.broadcast_to(w, y1.shape)[mask],
                               rtol=1e-14)
    # rows are independent: changing one row's o leaves the others
    o2 = o.copy()
    o2[2, 0] *= -3.0
    y2 = oracle.gated_rmsnorm(o2, z, w, 1e-6)
    np.testing.assert_array_equal(np.delete(y2.reshape(6, dv), 4, 0),
                                  np.delete(yw.reshape(6, dv), 4, 0))


# ---------------------------------------------------------------- phase-1 projection and norm
def test_linear_brute_force_and_closed_forms():
    r = rng(31)
    a = r.standard_normal((5, 7))
    w = r.standard_normal((4, 7))
    c = oracle.linear(a, w)
    brute = [[sum(a[m, k] * w[n, k] for k in range(7)) for n in range(4)] for m in range(5)]
    np.testing.assert_allclose(c, brute, rtol=1e-13, atol=1e-13)
    assert c.shape == (5, 4)
    # A = I picks the rows of W as columns; a rank-one A = u v^T gives u (W v)^T
    np.testing.assert_array_equal(oracle.linear(np.eye(7), w), w.T)
    u, v = r.standard_normal(5), r.standard_normal(7)
    np.testing.assert_allclose(oracle.linear(np.outer(u, v), w), np.outer(u, w @ v), rtol=1e-12)
    # zero columns appended to both operands (a K tail) change nothing
    a0 = np.concatenate([a, np.zeros((5, 9))], axis=1)
    w0 = np.concatenate([w, r.standard_normal((4, 9)) * 0], axis=1)
    np.testing.assert_array_equal(oracle.linear(a0, w0), c)


def test_rmsnorm_rows_closed_forms():
    # constant row 3 with eps = 7: 3 / sqrt(9 + 7) = 0.75; unit RMS at eps = 0; scale invariance
    x = np.full((2, 8), 3.0)
    np.testing.assert_allclose(oracle.rmsnorm_rows(x, np.full(8, 2.0), 7.0), 1.5, rtol=1e-15)
    r = rng(32)
    x = r.standard_normal((6, 64))
    y = oracle.rmsnorm_rows(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rmsnorm_rows(5.5 * x, np.ones(64), 0.0), y, rtol=1e-13)
    w = r.uniform(0.5, 2, 64)
    np.testing.assert_allclose(oracle.rmsnorm_rows(x, w, 0.0) / y, np.broadcast_to(w, y.shape),
                               rtol=1e-13)


def test_gate_activations_closed_forms():
    """softplus(0) = ln 2, softplus(ln 3) = ln 4, softplus(a) -> a for large a and -> e^a for very
    negative a; sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(-b) = 1 - sigmoid(b)."""
    a = np.array([0.0, math.log(3.0), 60.0, -60.0, 800.0])
    b = np.array([0.0, math.log(3.0), -2.5, 2.5, -800.0])
    g, beta = oracle.gate_activations(a, b)
    np.testing.assert_allclose(g[:2], [-math.log(2.0), -math.log(4.0)], rtol=1e-15)
    np.testing.assert_allclose(g[2], -60.0, rtol=1e-15)
    np.testing.assert_allclose(g[3], -math.exp(-60.0), rtol=1e-12)
    assert g[4] == -800.0 and np.all(g <= 0)
    np.testing.assert_allclose(beta[:2], [0.5, 0.75], rtol=1e-15)
    np.testing.assert_allclose(beta[2] + beta[3], 1.0, rtol=1e-15)
    assert beta[4] == 0.0
