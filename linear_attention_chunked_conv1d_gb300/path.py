"""One prefill pass of a GDN/KDA layer's hot path through the C ABI.

Order of the steps as on "glm5next_kda/prefill.rs" (Glm5NextKdaLayer::prefill_with_pad_fill)
and "split_prefill.rs" (prefill_phase1_conv1d_one per request, prefill_phase1_l2_batched, then
prefill_gdn_full_batched when all streams have one length, else the varlen call):

    conv1d + SiLU (per stream, carried conv state)  ->  L2 over the q|k heads  ->  recurrence

With bf16 activations and head dim 128 the whole pass is one launch (`fused`, the library's
la_prefill_front): the tensor-core recurrence computes its q, k, v tiles from the pre-conv rows
itself. Otherwise (and in `run_unfused`) the packed front-end output
[tokens][q heads | k heads | v heads] is handed to the recurrence as three strided views
(q, k, v), which is all the pages' split_widen step amounts to here.
This module only sequences the library calls; it holds no arithmetic.
"""
from __future__ import annotations

import math

import torch

from . import (conv1d_silu_l2_prefill, conv1d_silu_prefill, conv1d_silu_prefill_varlen,
               decode_step, decode_workspace_bytes, gate_activations, gdn_prefill_batched,
               gdn_prefill_varlen, gemm_bf16, kda_prefill, l2norm_heads, pointer_array,
               prefill_front, prefill_segmented, prefill_segmented_workspace_bytes,
               prefill_workspace_bytes, rmsnorm_rows)


class PrefillPass:
    """Buffers and state pointers for repeated passes over one packed batch on one device.

    `inputs` holds device tensors: x [T][cd], conv_w [cd][K], conv_state [B][K-1][cd],
    h [B][Hv][d][d] (fp32), g, beta, cu_seqlens, plus `lengths` (host list)."""

    def __init__(self, wl, inputs: dict, *, eps: float = 1e-6, pad_fill: float = 0.0):
        self.wl = wl
        self.inp = inputs
        self.eps = eps
        self.pad_fill = pad_fill
        x = inputs["x"]
        self.T = x.shape[0]
        self.lengths = list(inputs["lengths"])
        self.max_seqlen = max(self.lengths)
        dev = x.device
        self.conv_out = torch.empty_like(x)
        self.out = torch.empty(self.T, wl.Hv, wl.d, dtype=x.dtype, device=dev)
        B = wl.B
        self.conv_state_ptrs = pointer_array([inputs["conv_state"][s] for s in range(B)])
        self.h_ptrs = pointer_array([inputs["h"][s] for s in range(B)])
        nbytes = prefill_workspace_bytes(B, self.T, wl.Hk, wl.Hv, wl.d, wl.d, x.dtype)
        self.workspace = (torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes
                          else None)
        hk = wl.Hk * wl.d
        self.q = self.conv_out[:, :hk]
        self.k = self.conv_out[:, hk:2 * hk]
        self.v = self.conv_out[:, 2 * hk:]
        self.scale = 1.0 / math.sqrt(wl.d)
        self.can_fuse = x.dtype == torch.bfloat16 and wl.d == 128

    def front_end(self, stream=None):
        """conv1d + SiLU and the q|k L2 norm in one fused launch (bitwise equal to the two)."""
        wl, inp = self.wl, self.inp
        conv1d_silu_l2_prefill(self.conv_state_ptrs, inp["x"], inp["conv_w"], self.conv_out,
                               None if wl.B == 1 else inp["cu_seqlens"], l2_heads=2 * wl.Hk,
                               head_dim=wl.d, eps=self.eps, stream=stream)

    def front_end_unfused(self, stream=None):
        """The pages' two launches: conv_prefill, then l2 in place over q|k."""
        wl, inp = self.wl, self.inp
        if wl.B == 1:
            conv1d_silu_prefill(inp["conv_state"][0], inp["x"], inp["conv_w"], self.conv_out,
                                stream=stream)
        else:
            conv1d_silu_prefill_varlen(self.conv_state_ptrs, inp["x"], inp["conv_w"],
                                       self.conv_out, inp["cu_seqlens"], stream=stream)
        l2norm_heads(self.conv_out, 2 * wl.Hk, wl.d, eps=self.eps, stream=stream)

    def recurrence(self, stream=None):
        wl, inp = self.wl, self.inp
        d = wl.d
        common = dict(Hk=wl.Hk, Hv=wl.Hv, dk=d, dv=d, scale=self.scale, workspace=self.workspace,
                      stream=stream)
        if wl.variant == "kda":
            kda_prefill(self.h_ptrs, self.q, self.k, self.v, inp["g"], inp["beta"], self.out,
                        None if wl.B == 1 else inp["cu_seqlens"], max_seqlen=self.max_seqlen,
                        pad_fill=self.pad_fill, **common)
        elif wl.batched:
            gdn_prefill_batched(self.h_ptrs, self.q, self.k, self.v, inp["g"], inp["beta"],
                                self.out, B=wl.B, T=self.lengths[0], **common)
        else:
            gdn_prefill_varlen(self.h_ptrs, self.q, self.k, self.v, inp["g"], inp["beta"],
                               self.out, inp["cu_seqlens"], max_seqlen=self.max_seqlen, **common)

    def recurrence_segmented(self, segments, stream=None):
        """The recurrence of a single stream as a chunk-parallel scan (la_prefill_segmented)."""
        wl, inp = self.wl, self.inp
        assert wl.B == 1, "the segmented scan covers one stream"
        nbytes = prefill_segmented_workspace_bytes(self.T, wl.Hv, segments)
        if getattr(self, "_seg_ws", None) is None or self._seg_ws.numel() < nbytes:
            self._seg_ws = torch.empty(nbytes, dtype=torch.uint8, device=self.out.device)
        prefill_segmented(self.h_ptrs, self.q, self.k, self.v, inp["g"], inp["beta"], self.out,
                          Hk=wl.Hk, Hv=wl.Hv, dk=wl.d, dv=wl.d, kda=wl.variant == "kda",
                          segments=segments, scale=self.scale, workspace=self._seg_ws,
                          stream=stream)

    def fused(self, stream=None):
        """conv1d + SiLU + L2 + recurrence in one launch (bf16, head dim 128)."""
        wl, inp = self.wl, self.inp
        prefill_front(self.conv_state_ptrs, self.h_ptrs, inp["x"], inp["conv_w"], inp["g"],
                      inp["beta"], self.out, None if wl.batched or wl.B == 1 else inp["cu_seqlens"],
                      B=wl.B, Hk=wl.Hk, Hv=wl.Hv, dk=wl.d, dv=wl.d, kda=wl.variant == "kda",
                      max_seqlen=self.max_seqlen, l2_eps=self.eps, scale=self.scale,
                      pad_fill=self.pad_fill, workspace=self.workspace, stream=stream)

    def run_unfused(self, stream=None):
        self.front_end(stream)
        self.recurrence(stream)
        return self.out

    def run(self, stream=None):
        if self.can_fuse:
            self.fused(stream)
            return self.out
        return self.run_unfused(stream)


class DecodeStep:
    """One decode step of a GDN/KDA layer for B streams (one new token each) on one device,
    through la_decode_step. `inputs` as for PrefillPass, with x [B][cd] (row s = stream s)."""

    def __init__(self, wl, inputs: dict, *, eps: float = 1e-6):
        self.wl = wl
        self.inp = inputs
        self.eps = eps
        x = inputs["x"]
        B = wl.B
        assert x.shape[0] == B, "a decode step takes one token per stream"
        dev = x.device
        self.out = torch.empty(B, wl.Hv, wl.d, dtype=x.dtype, device=dev)
        self.conv_state_ptrs = pointer_array([inputs["conv_state"][s] for s in range(B)])
        self.h_ptrs = pointer_array([inputs["h"][s] for s in range(B)])
        nbytes = decode_workspace_bytes(B, wl.Hk, wl.Hv, wl.d, wl.d, x.dtype)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.scale = 1.0 / math.sqrt(wl.d)

    def run(self, stream=None):
        wl, inp = self.wl, self.inp
        decode_step(self.conv_state_ptrs, self.h_ptrs, inp["x"], inp["conv_w"], inp["g"],
                    inp["beta"], self.out, Hk=wl.Hk, Hv=wl.Hv, dk=wl.d, dv=wl.d,
                    kda=wl.variant == "kda", l2_eps=self.eps, scale=self.scale,
                    workspace=self.workspace, stream=stream)
        return self.out


class Phase1:
    """Phase 1 of a layer over the stacked hidden rows ("split_prefill.rs",
    prefill_phase1_proj_batched: norm, QKVZ, gates), through the library:
    rmsnorm_rows -> three projection GEMMs (q|k|v, z, gate pre-activations a|b) -> gate
    activations. Weights are the caller's ([out][in] bf16); outputs are device tensors:
    x [t][cd] (the conv input), z [t][Hv*dv], g (fp32 [t][Hv] or [t][Hv*dk]), beta [t][Hv]."""

    def __init__(self, wl, norm_w, w_qkv, w_z, w_ab, *, eps=1e-6):
        self.wl, self.norm_w, self.w_qkv, self.w_z, self.w_ab, self.eps = (
            wl, norm_w, w_qkv, w_z, w_ab, eps)
        self.na = wl.Hv * (wl.d if wl.variant == "kda" else 1)

    def run(self, hidden, stream=None):
        y = rmsnorm_rows(hidden, self.norm_w, eps=self.eps, stream=stream)
        x = gemm_bf16(y, self.w_qkv, stream=stream)
        z = gemm_bf16(y, self.w_z, stream=stream)
        n_ab = self.w_ab.shape[0]  # rows padded to 16 bytes (the GEMM's output stride rule)
        ab = torch.empty(y.shape[0], (n_ab + 7) // 8 * 8, dtype=y.dtype, device=y.device)[:, :n_ab]
        gemm_bf16(y, self.w_ab, ab, stream=stream)
        g, beta = gate_activations(ab, self.na, stream=stream)
        return dict(y=y, x=x, z=z, ab=ab, g=g, beta=beta)


class StreamedPrefill:
    """Prefill steps fed from pinned host memory and read back to it, pipelined over three
    streams: the host->device copy of step i+1 and the device->host copy of step i-1 overlap
    the compute of step i. Two sets of device inputs and outputs alternate; the carried conv and
    h states are shared and advance in step order on the compute stream.

    `mode`: "split" (fused conv+L2, then the recurrence), "fused" (la_prefill_front) or "seg"
    (fused conv+L2, then the segmented recurrence with `segments` pieces, one stream)."""

    def __init__(self, wl, inputs: dict, *, mode="split", segments=1, compute_stream=None):
        self.mode, self.segments = mode, segments
        dev = inputs["x"].device
        self.passes = []
        for _ in range(2):
            inp = dict(inputs)
            for name in ("x", "g", "beta"):
                inp[name] = torch.empty_like(inputs[name])
            self.passes.append(PrefillPass(wl, inp))
        self.compute = compute_stream or torch.cuda.current_stream(dev)
        self.copy_in = torch.cuda.Stream(dev)
        self.copy_out = torch.cuda.Stream(dev)
        self.copied = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.drained = [torch.cuda.Event() for _ in range(2)]

    def _run(self, p):
        if self.mode == "fused":
            p.fused(self.compute)
        elif self.mode == "seg":
            p.front_end(self.compute)
            p.recurrence_segmented(self.segments, self.compute)
        else:
            p.run_unfused(self.compute)

    def step(self, i, x_h, g_h, beta_h, out_h):
        """Step i: inputs from the pinned host tensors, the output into out_h (all queued)."""
        b = i % 2
        p = self.passes[b]
        with torch.cuda.stream(self.copy_in):
            self.copy_in.wait_event(self.computed[b])  # step i-2 is done with these inputs
            p.inp["x"].copy_(x_h, non_blocking=True)
            p.inp["g"].copy_(g_h, non_blocking=True)
            p.inp["beta"].copy_(beta_h, non_blocking=True)
            self.copied[b].record(self.copy_in)
        self.compute.wait_event(self.copied[b])
        self.compute.wait_event(self.drained[b])  # step i-2's output has been read back
        self._run(p)
        self.computed[b].record(self.compute)
        with torch.cuda.stream(self.copy_out):
            self.copy_out.wait_event(self.computed[b])
            out_h.copy_(p.out, non_blocking=True)
            self.drained[b].record(self.copy_out)

    def start(self, event):
        """Make every stream of the pipeline start after `event` (recorded by the caller)."""
        for st in (self.compute, self.copy_in, self.copy_out):
            st.wait_event(event)

    def finish(self):
        """Make the compute stream wait for the last copies back (then record on it)."""
        self.compute.wait_event(self.drained[0])
        self.compute.wait_event(self.drained[1])
