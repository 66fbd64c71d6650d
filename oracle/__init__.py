"""fp64 CPU oracle for the chunked gated-delta-rule prefill path — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. The product library (``linear_attention_chunked_conv1d_gb300``) never
imports, links or calls it, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain sequential C, fp64, one host thread per
(stream, v-head) unit), except the phase-1 projection and its row norm (``linear``,
``rmsnorm_rows``), written here in fp64 numpy around one matrix product; this module marshals
numpy float64 arrays into the C code and composes the steps in the order the pages launch them ("glm5next_kda/prefill.rs",
``Glm5NextKdaLayer::prefill_with_pad_fill``: conv_prefill -> l2 -> chunk_prepare/chunk_scan).

Reading of the pages (where they are silent): activations produced by the front end are
stored in the activation dtype before the next step reads them — the pages write the conv
output into a workspace buffer (``ws.conv_out``) and run the L2 norm in place on that
buffer — so ``front_end`` rounds the conv output and the normalised q|k to ``act_dtype``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_D = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (fp contraction off, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.or_conv1d_silu.argtypes = [_D, _D, _D, _D, _D, _D, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_long, ctypes.c_long]
            lib.or_conv1d_silu.restype = None
            lib.or_l2norm_heads.argtypes = [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_long, ctypes.c_double]
            lib.or_l2norm_heads.restype = None
            lib.or_gated_delta_varlen.argtypes = [
                ctypes.POINTER(_D), _D, _D, _D, _D, _D, _D, ctypes.POINTER(ctypes.c_int32),
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_double,
                ctypes.c_int]
            lib.or_gated_delta_varlen.restype = None
            lib.or_gated_rmsnorm.argtypes = [_D, _D, _D, _D, ctypes.c_long, ctypes.c_int,
                                             ctypes.c_double]
            lib.or_gated_rmsnorm.restype = None
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def conv1d_silu(state, x, w, bias=None):
    """Causal depthwise conv1d + SiLU over one stream.

    state [K-1][C] (oldest row first), x [t][C], w [C][K] (tap K-1 multiplies the current
    token), bias [C] or None. Returns (out [t][C], new_state [K-1][C])."""
    lib = _load()
    x = _f64(x)
    w = _f64(w)
    C, K = w.shape
    t = x.shape[0]
    state = _f64(state).reshape(K - 1, C) if K > 1 else np.zeros((0, C))
    out = np.zeros((t, C))
    new_state = np.zeros((K - 1, C))
    b = _f64(bias) if bias is not None else None
    lib.or_conv1d_silu(_p(state) if K > 1 else None, _p(x) if t else None, _p(w),
                       _p(b) if b is not None else None, _p(out) if t else None,
                       _p(new_state) if K > 1 else None, t, C, K, C, C)
    return out, new_state


def conv1d_silu_varlen(states, x, w, cu_seqlens, bias=None):
    """conv1d_silu per stream of a packed batch; states [B][K-1][C]. Returns (out, new_states)."""
    x = _f64(x)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = np.zeros_like(x)
    new_states = np.array(_f64(states), copy=True)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        out[a:b], new_states[s] = conv1d_silu(new_states[s], x[a:b], w, bias)
    return out, new_states


def l2norm_heads(x, n_heads, head_dim, eps):
    """Per (token, head) L2 norm of the first n_heads*head_dim channels of x [t][C] (a copy)."""
    lib = _load()
    y = np.array(_f64(x), copy=True)
    t, C = y.shape
    if t:
        lib.or_l2norm_heads(_p(y), t, n_heads, head_dim, C, float(eps))
    return y


def gated_rmsnorm(o, z, w, eps):
    """Gated RMSNorm per row of the last axis (dv): o / sqrt(mean(o^2) + eps) * w * SiLU(z).
    o, z [..., dv] (same shape), w [dv]. Returns a new array."""
    lib = _load()
    o = np.ascontiguousarray(_f64(o))
    z = np.ascontiguousarray(_f64(z))
    w = np.ascontiguousarray(_f64(w))
    assert o.shape == z.shape and w.shape == (o.shape[-1],)
    y = np.empty_like(o)
    dv = o.shape[-1]
    n = o.size // dv if dv else 0
    if n:
        lib.or_gated_rmsnorm(_p(o), _p(z), _p(w), _p(y), n, dv, float(eps))
    return y


def linear(a, w):
    """Phase-1 projection of a batch of rows ("split_prefill.rs",
    LayerSplitPrefill::prefill_phase1_proj_batched: the QKVZ and gate projections of the
    normalised hidden rows): C = A W^T in fp64, with A [M][K] and W [N][K] in the [out][in]
    layout of a linear layer. The matrix product is the library primitive of this step."""
    return _f64(a) @ _f64(w).T


def rmsnorm_rows(x, w, eps):
    """The norm of phase 1: y = x / sqrt(mean(x^2) + eps) * w per row (fp64)."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(w)


def gate_activations(a, b):
    """The gates of phase 1 from their projections: g = -softplus(a) = -log(1 + e^a) (the
    log-decay, <= 0) and beta = sigmoid(b) = 1 / (1 + e^-b), in fp64. This is the plain reading
    of "gates" in prefill_phase1_proj_batched, and the transform of the synthetic input recipe."""
    a, b = _f64(a), _f64(b)
    return -np.logaddexp(0.0, a), 1.0 / (1.0 + np.exp(-b))


def gated_delta(h_states, q, k, v, g, beta, cu_seqlens, *, scale, per_channel=False,
                threads=None):
    """Token-by-token gated delta rule over packed streams.

    h_states [B][Hv][dk][dv] (H = S^T), q/k [T][Hk][dk], v [T][Hv][dv], g [T][Hv] (GDN) or
    [T][Hv][dk] (KDA), beta [T][Hv], cu_seqlens [B+1]. Returns (out [T][Hv][dv], new states).
    """
    lib = _load()
    h = np.array(_f64(h_states), copy=True)
    B, Hv, dk, dv = h.shape
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    T = v.shape[0]
    Hk = q.shape[1]
    q = q.reshape(T, Hk * dk)
    k = k.reshape(T, Hk * dk)
    v = v.reshape(T, Hv * dv)
    g = _f64(g)
    beta = _f64(beta)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    assert cu.shape == (B + 1,)
    out = np.zeros((T, Hv, dv))
    if T == 0:
        return out, h
    ptrs = (_D * B)(*[ctypes.cast(h[s].ctypes.data, _D) for s in range(B)])
    nthr = threads if threads is not None else (os.cpu_count() or 1)
    lib.or_gated_delta_varlen(ptrs, _p(q), _p(k), _p(v), _p(g), _p(beta), _p(out),
                              cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, Hk, Hv,
                              dk, dv, Hk * dk, Hk * dk, Hv * dv, 1 if per_channel else 0,
                              float(scale), int(nthr))
    return out, h


def round_to(a, act_dtype: str):
    """Round fp64 values to the activation dtype ('f32' or 'bf16', nearest-even) and widen."""
    a = _f64(a)
    if act_dtype == "f32":
        return a.astype(np.float32).astype(np.float64)
    if act_dtype == "bf16":
        import torch
        return torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    raise ValueError(act_dtype)


def front_end(x, conv_w, conv_states, cu_seqlens, *, Hk, Hv, dk, dv, eps, act_dtype,
              bias=None):
    """conv1d+SiLU per stream, then L2 per head over the q|k channels.

    x [T][cd] with cd = 2*Hk*dk + Hv*dv laid out [q heads | k heads | v heads]. Returns
    (q [T][Hk][dk], k [T][Hk][dk], v [T][Hv][dv], new conv states); each stored step is
    rounded to act_dtype as the pages' buffers are."""
    conv_out, new_states = conv1d_silu_varlen(conv_states, x, conv_w, cu_seqlens, bias)
    conv_out = round_to(conv_out, act_dtype)
    normed = l2norm_heads(conv_out, 2 * Hk, dk, eps)
    normed = round_to(normed, act_dtype)
    T = x.shape[0]
    q = normed[:, :Hk * dk].reshape(T, Hk, dk)
    k = normed[:, Hk * dk:2 * Hk * dk].reshape(T, Hk, dk)
    v = normed[:, 2 * Hk * dk:].reshape(T, Hv, dv)
    return q, k, v, new_states
