"""Shared helpers of the GPU parity tests: run the oracle on the same inputs, compare."""
import numpy as np
import torch

import oracle

# Acceptance bars (max abs error on outputs; relative Frobenius error on final states).
TOL = {"bf16": dict(out=2e-3, state=1e-3), "f32": dict(out=1e-5, state=1e-5)}


def f64(t) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def act_name(dtype) -> str:
    return "bf16" if dtype == torch.bfloat16 else "f32"


def oracle_front(x, conv_w, conv_state, lengths, Hk, Hv, d, eps, act):
    cu = np.concatenate([[0], np.cumsum(lengths)])
    return oracle.front_end(f64(x), f64(conv_w), f64(conv_state), cu, Hk=Hk, Hv=Hv, dk=d, dv=d,
                            eps=eps, act_dtype=act)


def oracle_recurrence(h, q, k, v, g, beta, lengths, scale, kda, heads=None):
    """Oracle over all v-heads, or over the listed v-heads only (each with its own k-head)."""
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v, g, beta, h = (f64(a) if torch.is_tensor(a) else a for a in (q, k, v, g, beta, h))
    if heads is not None:
        Hk, Hv = q.shape[1], v.shape[1]
        kh = [j * Hk // Hv for j in heads]
        q, k = q[:, kh], k[:, kh]
        v, g, beta, h = v[:, heads], g[:, heads], beta[:, heads], h[:, heads]
    return oracle.gated_delta(h, q, k, v, g, beta, cu, scale=scale, per_channel=kda)


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b)))) if np.size(a) else 0.0


def rel_frob(a, ref) -> float:
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / den) if den > 0 else float(np.linalg.norm(a))


def bf16_ulp_diff(gpu: torch.Tensor, ref: np.ndarray) -> int:
    """Max distance in bf16 ulps between a bf16 tensor and fp64 reference values rounded to bf16."""
    r = torch.from_numpy(np.ascontiguousarray(ref)).to(torch.bfloat16)
    a = gpu.detach().cpu().contiguous().view(torch.int16).to(torch.int32)
    b = r.view(torch.int16).to(torch.int32)
    # map sign-magnitude bf16 bit patterns onto a monotone integer line
    a = torch.where(a < 0, -(a & 0x7FFF), a)
    b = torch.where(b < 0, -(b & 0x7FFF), b)
    return int((a - b).abs().max()) if a.numel() else 0
