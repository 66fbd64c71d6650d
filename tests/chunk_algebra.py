"""Test-only fp64 restatement of the chunked (WY) form that the CUDA kernels compute.

It exists to pin the algebra, not to serve as the oracle: the tests require it to equal the
token-by-token oracle to 1e-10, so a sign, index or decay-reference mistake in the chunk
formulas shows up here on the CPU before any kernel runs. Per chunk of C tokens, with gc the
inclusive cumulative log-gate (one value per k-channel; GDN broadcasts it):
    A[t][i] = beta_t sum_c K[t][c] K[i][c] e^{gc[t][c] - gc[i][c]}   (i < t)
    P[t][i] =        sum_c Q[t][c] K[i][c] e^{gc[t][c] - gc[i][c]}   (i <= t)
    U'      = (I + A)^{-1} diag(beta) (V - (K (.) e^{gc}) H)
    O       = scale ((Q (.) e^{gc}) H + P U')
    H      <- diag(e^{gc_L}) H + (K (.) e^{gc_L - gc})^T U'
"""
import numpy as np
from scipy.linalg import solve_triangular


def chunked_unit(H0, q, k, v, g, beta, *, scale, C=64):
    """One (stream, v-head) unit. H0 [dk][dv]; q, k [T][dk]; v [T][dv]; g [T] or [T][dk]."""
    H = np.array(H0, dtype=np.float64, copy=True)
    T, dk = k.shape
    g = np.asarray(g, dtype=np.float64)
    if g.ndim == 1:
        g = np.repeat(g[:, None], dk, axis=1)
    out = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        K, Q, V, b = k[sl], q[sl], v[sl], beta[sl]
        n = K.shape[0]
        gc = np.cumsum(g[sl], axis=0)
        D = np.exp(gc[:, None, :] - gc[None, :, :])
        A = np.tril(b[:, None] * np.einsum("tc,ic,tic->ti", K, K, D), -1)
        P = np.tril(np.einsum("tc,ic,tic->ti", Q, K, D))
        R = b[:, None] * (V - (K * np.exp(gc)) @ H)
        U = solve_triangular(np.eye(n) + A, R, lower=True, unit_diagonal=True)
        out[sl] = scale * ((Q * np.exp(gc)) @ H + P @ U)
        H = np.exp(gc[-1])[:, None] * H + (K * np.exp(gc[-1][None, :] - gc)).T @ U
    return out, H
