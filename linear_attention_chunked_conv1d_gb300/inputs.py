"""Seeded synthetic inputs for the prefill path (shared by tests, bench and smoke).

This module draws random numbers and applies the input recipe only (gate = -softplus(N(0,1)),
beta = sigmoid(N(0,1)), casts); it holds none of the method's arithmetic. The same host
tensors feed the CUDA path and the oracle.

Recipe (one torch.Generator seeded with `seed`, fixed draw order): stream lengths, x, conv w,
conv state, h state, gate pre-activation, beta pre-activation. N(0, s) takes s as the standard
deviation: x ~ N(0, 1), conv w ~ N(0, 0.25), h ~ N(0, 0.02); carried conv state ~ N(0, 1) where
the workload carries one, zeros otherwise.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    variant: str           # "gdn" (scalar gate per v-head) or "kda" (gate per k-channel)
    B: int                 # streams
    Hk: int                # q/k heads
    Hv: int                # v heads
    d: int                 # head dim (dk = dv)
    lengths: str           # "fixed:T", "uniform:lo:hi", "loguniform:lo:hi:total"
    dtype: str = "bf16"    # activation dtype: "bf16" or "f32"
    conv_kernel: int = 4
    conv_state: str = "zero"   # "zero" or "randn"
    h_state: str = "zero"      # "zero" or "randn" (std h_std)
    h_std: float = 0.02
    x_std: float = 1.0
    w_std: float = 0.25
    batched: bool = False      # equal-length streams through the batched call
    mode: str = "prefill"      # "prefill", "decode" (one new token per stream, lengths fixed:1)
                               # or "proj" (the phase-1 projection GEMM of the stacked tokens)
    hidden: int = 0            # proj: width of the hidden rows (the GEMM's K)

    @property
    def cd(self) -> int:
        return 2 * self.Hk * self.d + self.Hv * self.d

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the path, by what they are.
WORKLOADS = {
    # GDN single stream, T = 100 (not a multiple of the chunk), 4 heads, d = 64, fp32, zero states
    "gdn_t100_h4_d64_f32": Workload("gdn_t100_h4_d64_f32", "gdn", 1, 4, 4, 64, "fixed:100",
                                    dtype="f32"),
    # GDN batched, 8 equal streams x 2048 tokens, 16 heads, d = 128, bf16, h ~ N(0, 0.02)
    "gdn_batched_8x2048_h16_d128": Workload("gdn_batched_8x2048_h16_d128", "gdn", 8, 16, 16, 128,
                                            "fixed:2048", h_state="randn", batched=True),
    # GDN varlen, 32 streams, lengths U[1, 8192], 16 q/k heads shared by 32 v heads, d = 128
    "gdn_varlen_32_hk16_hv32_d128": Workload("gdn_varlen_32_hk16_hv32_d128", "gdn", 32, 16, 32,
                                             128, "uniform:1:8192", conv_state="randn",
                                             h_state="randn"),
    # KDA single stream, T = 4096 from a carried nonzero state, 32 heads, d = 128
    "kda_t4096_h32_d128": Workload("kda_t4096_h32_d128", "kda", 1, 32, 32, 128, "fixed:4096",
                                   conv_state="randn", h_state="randn"),
    # KDA varlen, 64 streams, log-uniform lengths in [16, 16384] summing to 262144, full front end
    "kda_varlen_64_h32_d128": Workload("kda_varlen_64_h32_d128", "kda", 64, 32, 32, 128,
                                       "loguniform:16:16384:262144", conv_state="randn",
                                       h_state="randn"),
}

# Decode steps (one token for each of 256 streams, carried states), the step after a prefill.
DECODE_WORKLOADS = {
    # GDN, 16 q/k heads shared by 32 v heads, d = 128, as the GDN varlen prefill
    "gdn_decode_256_hk16_hv32_d128": Workload("gdn_decode_256_hk16_hv32_d128", "gdn", 256, 16, 32,
                                              128, "fixed:1", conv_state="randn",
                                              h_state="randn", mode="decode"),
    # KDA, 32 heads, d = 128, as the KDA prefills
    "kda_decode_256_h32_d128": Workload("kda_decode_256_h32_d128", "kda", 256, 32, 32, 128,
                                        "fixed:1", conv_state="randn", h_state="randn",
                                        mode="decode"),
}


def loguniform_lengths(u: np.ndarray, lo: int, hi: int, total: int) -> list[int]:
    """Lengths e^u (u ~ U(ln lo, ln hi)) rescaled to sum to `total`, clamped to [lo, hi] with the
    remainder redistributed over the unclamped streams, rounded half-even, and the final unit
    difference put on the longest unclamped stream."""
    L = np.exp(u.astype(np.float64))
    clamped = np.zeros(L.shape, dtype=bool)
    for _ in range(200):
        free = ~clamped
        remaining = total - L[clamped].sum()
        L[free] *= remaining / L[free].sum()
        newly = free & ((L < lo) | (L > hi))
        if not newly.any():
            break
        L = np.clip(L, lo, hi)
        clamped |= newly
    Li = np.rint(L).astype(np.int64)
    free_idx = np.where(~clamped)[0]
    pick = free_idx[np.argmax(Li[free_idx])] if len(free_idx) else int(np.argmax(Li))
    Li[pick] += total - Li.sum()
    return [int(v) for v in Li]


def draw_lengths(wl: Workload, gen: torch.Generator) -> list[int]:
    kind, *args = wl.lengths.split(":")
    if kind == "fixed":
        return [int(args[0])] * wl.B
    if kind == "uniform":
        lo, hi = int(args[0]), int(args[1])
        return [int(v) for v in torch.randint(lo, hi + 1, (wl.B,), generator=gen)]
    if kind == "loguniform":
        lo, hi, total = int(args[0]), int(args[1]), int(args[2])
        u = torch.rand(wl.B, generator=gen, dtype=torch.float64) * (math.log(hi) - math.log(lo))
        return loguniform_lengths((u + math.log(lo)).numpy(), lo, hi, total)
    if kind == "list":
        return [int(v) for v in args[0].split(",")]
    raise ValueError(wl.lengths)


def make_inputs(wl: Workload, device="cpu", seed: int = 0) -> dict:
    """All inputs of one pass of the path for workload `wl`, drawn on `device`.

    Lengths are always drawn on the CPU generator so that they do not depend on the device."""
    gcpu = torch.Generator("cpu")
    gcpu.manual_seed(seed)
    lengths = draw_lengths(wl, gcpu)
    gen = gcpu if str(device) == "cpu" else torch.Generator(device)
    if gen is not gcpu:
        gen.manual_seed(seed)
    T = sum(lengths)
    cd, K, d = wl.cd, wl.conv_kernel, wl.d
    act = wl.torch_dtype
    f32 = torch.float32

    def randn(*shape, std=1.0):
        return torch.randn(*shape, generator=gen, device=device, dtype=f32) * std

    x = randn(T, cd, std=wl.x_std).to(act)
    conv_w = randn(cd, K, std=wl.w_std).to(act)
    conv_state = randn(wl.B, K - 1, cd).to(act)
    if wl.conv_state == "zero":
        conv_state.zero_()
    h = randn(wl.B, wl.Hv, d, d, std=wl.h_std)
    if wl.h_state == "zero":
        h.zero_()
    gshape = (T, wl.Hv, d) if wl.variant == "kda" else (T, wl.Hv)
    g = -torch.nn.functional.softplus(randn(*gshape))
    beta = torch.sigmoid(randn(T, wl.Hv))
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32, device=device)
    return dict(lengths=lengths, cu_seqlens=cu, x=x, conv_w=conv_w, conv_state=conv_state,
                h=h, g=g, beta=beta)


def recurrence_inputs(B_lengths, Hk, Hv, d, *, kda=False, dtype="bf16", seed=0, h_std=0.02,
                      device="cpu") -> dict:
    """Direct q/k/v inputs (no front end) for recurrence-only tests: q, k ~ N(0, 1/sqrt(d)) so
    that their rows have norm close to 1, as the front end's L2 norm leaves them; v ~ N(0, 0.5)."""
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    T = sum(B_lengths)
    act = torch.bfloat16 if dtype == "bf16" else torch.float32
    f32 = torch.float32
    q = torch.randn(T, Hk, d, generator=gen, dtype=f32) / math.sqrt(d)
    k = torch.randn(T, Hk, d, generator=gen, dtype=f32) / math.sqrt(d)
    v = torch.randn(T, Hv, d, generator=gen, dtype=f32) * 0.5
    h = torch.randn(len(B_lengths), Hv, d, d, generator=gen, dtype=f32) * h_std
    gshape = (T, Hv, d) if kda else (T, Hv)
    g = -torch.nn.functional.softplus(torch.randn(*gshape, generator=gen, dtype=f32))
    beta = torch.sigmoid(torch.randn(T, Hv, generator=gen, dtype=f32))
    cu = torch.tensor([0] + list(np.cumsum(B_lengths)), dtype=torch.int32)
    out = dict(q=q.to(act), k=k.to(act), v=v.to(act), h=h, g=g, beta=beta, cu_seqlens=cu,
               lengths=list(B_lengths))
    return {k_: (v_.to(device) if torch.is_tensor(v_) else v_) for k_, v_ in out.items()}

# Phase-1 projection (QKVZ) of the stacked tokens of the batched GDN prefill: 16384 tokens,
# hidden 2048 -> q | k | v | z = 4 x 16 heads x 128 = 8192 outputs, bf16, random weights.
PROJ_WORKLOADS = {
    "proj_qkvz_16384x2048x8192": Workload("proj_qkvz_16384x2048x8192", "gdn", 8, 16, 16, 128,
                                          "fixed:2048", mode="proj", hidden=2048),
}
