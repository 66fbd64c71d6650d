"""GB300-native chunked gated-delta-rule prefill (GDN / KDA) with a causal conv1d front end.

Thin Python binding of the C ABI in ``include/linattn.h`` (``liblinattn.so``): every function
here only marshals torch CUDA tensors into raw device pointers, sizes and the current CUDA
stream, then calls the C entry point of the same name. All arithmetic runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback, and importing fails loudly when the library
has not been built (``python -m linear_attention_chunked_conv1d_gb300.build``).
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB_PATH

__all__ = [
    "LinAttnError", "LA_F32", "LA_BF16", "abi_version", "last_error", "device_status",
    "conv1d_silu_prefill", "conv1d_silu_prefill_varlen", "conv1d_silu_l2_prefill",
    "l2norm_heads",
    "prefill_workspace_bytes", "gdn_prefill_batched", "gdn_prefill_varlen",
    "gdn_prefill_varlen_noalloc", "kda_prefill",
    "pointer_array", "library_path",
]

LA_OK, LA_ERR_ARG, LA_ERR_COUNT, LA_ERR_UNSUPPORTED, LA_ERR_CUDA = 0, 1, 2, 3, 4
LA_F32, LA_BF16 = 0, 1
LA_DEV_BAD_SEQLENS, LA_DEV_TIMEOUT = 1, 2
_CODES = {LA_ERR_ARG: "LA_ERR_ARG", LA_ERR_COUNT: "LA_ERR_COUNT",
          LA_ERR_UNSUPPORTED: "LA_ERR_UNSUPPORTED", LA_ERR_CUDA: "LA_ERR_CUDA"}


class LinAttnError(RuntimeError):
    """A linattn call returned a non-zero status; ``code`` holds it."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"{_CODES.get(code, code)}: {msg}")
        self.code = code


_u64, _i64, _i32, _f32, _vp, _sz = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t)

_SIGS = {
    "la_abi_version": ([], ctypes.c_int),
    "la_last_error": ([], ctypes.c_char_p),
    "la_device_status": ([_u64], ctypes.c_int),
    "la_conv1d_silu_prefill": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i64,
                                _i32, _u64], ctypes.c_int),
    "la_conv1d_silu_prefill_varlen": ([_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                       _i32, _i64, _i64, _i32, _u64], ctypes.c_int),
    "la_l2norm_heads": ([_vp, _i32, _i32, _i32, _i64, _f32, _i32, _u64], ctypes.c_int),
    "la_conv1d_silu_l2_prefill": ([_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                   _i32, _i32, _f32, _i64, _i64, _i32, _u64], ctypes.c_int),
    "la_prefill_workspace_bytes": ([_i32, _i32, _i32, _i32, _i32, _i32, _i32], _sz),
    "la_gdn_prefill_batched": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                _i32, _i32, _i64, _i64, _i64, _f32, _i32, _vp, _sz, _u64],
                               ctypes.c_int),
    "la_gdn_prefill_varlen": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                               _i32, _i32, _i32, _i32, _i64, _i64, _i64, _f32, _i32, _vp, _sz,
                               _u64], ctypes.c_int),
    "la_gdn_prefill_varlen_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                       _i32, _i32, _i32, _i32, _i32, _i32, _i64, _i64, _i64,
                                       _f32, _u64], ctypes.c_int),
    "la_kda_prefill": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                        _i32, _i32, _i32, _i64, _i64, _i64, _f32, _f32, _i32, _vp, _sz, _u64],
                       ctypes.c_int),
    "la_prefill_front": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                          _i32, _i32, _i32, _i32, _i32, _i64, _f32, _f32, _f32, _vp, _vp, _f32,
                          _i32, _i32, _vp, _sz, _u64], ctypes.c_int),
    "la_gated_rmsnorm": ([_vp, _vp, _vp, _vp, _i32, _i32, _i32, _f32, _i32, _u64], ctypes.c_int),
    "la_gemm_bf16": ([_vp, _vp, _vp, _i32, _i32, _i32, _i64, _i64, _i64, _u64], ctypes.c_int),
    "la_prefill_segmented_workspace_bytes": ([_i32, _i32, _i32], _sz),
    "la_prefill_segmented": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                              _i32, _i64, _i64, _i64, _f32, _i32, _i32, _i32, _vp, _sz, _u64],
                             ctypes.c_int),
    "la_rmsnorm_rows": ([_vp, _vp, _vp, _i32, _i32, _i64, _i64, _f32, _u64], ctypes.c_int),
    "la_gate_activations": ([_vp, _i64, _i32, _i32, _i32, _vp, _vp, _u64], ctypes.c_int),
    "la_decode_workspace_bytes": ([_i32, _i32, _i32, _i32, _i32, _i32], _sz),
    "la_decode_step": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                        _i32, _i32, _i64, _f32, _f32, _i32, _i32, _vp, _sz, _u64], ctypes.c_int),
}

_lib = None


def library_path() -> str:
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"linattn CUDA library not built ({LIB_PATH} missing); run "
                "`python -m linear_attention_chunked_conv1d_gb300.build` — there is no fallback")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _check(rc: int) -> None:
    if rc != LA_OK:
        raise LinAttnError(rc, last_error())


def abi_version() -> int:
    return _load().la_abi_version()


def last_error() -> str:
    return _load().la_last_error().decode()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def device_status(stream=None) -> int:
    """Synchronise the stream and return (then clear) the device status flags (LA_DEV_*)."""
    return _load().la_device_status(_stream(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError(f"activation dtype {t.dtype}: expected float32 or bfloat16")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _row_stride(t: torch.Tensor) -> int:
    return t.stride(0)


def pointer_array(tensors, device=None) -> torch.Tensor:
    """Device array of the data pointers of `tensors` (h-state / conv-state lists), stored as
    int64 (the same 64 bits the C ABI reads as uint64_t)."""
    ptrs = [t.data_ptr() for t in tensors]
    dev = device if device is not None else tensors[0].device
    return torch.tensor(ptrs, dtype=torch.int64, device=dev)


def conv1d_silu_prefill(conv_state, x, w, out, *, t=None, bias=None, max_tokens=None,
                        stream=None) -> None:
    """Causal conv1d + SiLU over one stream, advancing conv_state [K-1][C] in place.

    x, out: [t][stride] (the first C = w.shape[0] channels are used); w [C][K]."""
    t = x.shape[0] if t is None else t
    C, K = w.shape
    _check(_load().la_conv1d_silu_prefill(
        _ptr(conv_state), _ptr(x), _ptr(w), _ptr(bias), _ptr(out), t,
        max_tokens if max_tokens is not None else t, C, K, _row_stride(x), _row_stride(out),
        _dtype_code(x), _stream(stream)))


def conv1d_silu_prefill_varlen(conv_state_ptrs, x, w, out, cu_seqlens, *, bias=None,
                               total_tokens=None, max_tokens=None, stream=None) -> None:
    """conv1d_silu_prefill over B packed streams; conv_state_ptrs is a device uint64 array."""
    B = cu_seqlens.shape[0] - 1
    total = x.shape[0] if total_tokens is None else total_tokens
    C, K = w.shape
    _check(_load().la_conv1d_silu_prefill_varlen(
        _ptr(conv_state_ptrs), _ptr(x), _ptr(w), _ptr(bias), _ptr(out), _ptr(cu_seqlens), B,
        total, max_tokens if max_tokens is not None else total, C, K, _row_stride(x),
        _row_stride(out), _dtype_code(x), _stream(stream)))


def conv1d_silu_l2_prefill(conv_state_ptrs, x, w, out, cu_seqlens=None, *, l2_heads, head_dim,
                           eps=1e-6, bias=None, total_tokens=None, max_tokens=None,
                           stream=None) -> None:
    """Fused conv1d + SiLU + per-head L2 over the first l2_heads*head_dim channels (one pass)."""
    B = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    total = x.shape[0] if total_tokens is None else total_tokens
    C, K = w.shape
    _check(_load().la_conv1d_silu_l2_prefill(
        _ptr(conv_state_ptrs), _ptr(x), _ptr(w), _ptr(bias), _ptr(out), _ptr(cu_seqlens), B,
        total, max_tokens if max_tokens is not None else total, C, K, l2_heads, head_dim,
        float(eps), _row_stride(x), _row_stride(out), _dtype_code(x), _stream(stream)))


def l2norm_heads(x, n_heads, head_dim, *, eps=1e-6, t=None, stream=None) -> None:
    """In-place L2 norm of each (token, head) over the first n_heads*head_dim channels."""
    t = x.shape[0] if t is None else t
    _check(_load().la_l2norm_heads(_ptr(x), t, n_heads, head_dim, _row_stride(x), float(eps),
                                   _dtype_code(x), _stream(stream)))


def prefill_workspace_bytes(B, total_tokens, Hk, Hv, dk, dv, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (LA_BF16 if dtype == torch.bfloat16 else LA_F32)
    return int(_load().la_prefill_workspace_bytes(B, total_tokens, Hk, Hv, dk, dv, code))


def gdn_prefill_batched(h_state_ptrs, q, k, v, g, beta, out, *, B, T, Hk, Hv, dk, dv,
                        scale=None, max_tokens=None, workspace=None, stream=None) -> None:
    """GDN over B equal-length streams of T tokens; states updated through h_state_ptrs."""
    scale = 1.0 / math.sqrt(dk) if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_load().la_gdn_prefill_batched(
        _ptr(h_state_ptrs), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(out), B, T,
        max_tokens if max_tokens is not None else B * T, Hk, Hv, dk, dv, _row_stride(q),
        _row_stride(k), _row_stride(v), float(scale), _dtype_code(q), _ptr(workspace), ws_bytes,
        _stream(stream)))


def gdn_prefill_varlen(h_state_ptrs, q, k, v, g, beta, out, cu_seqlens, *, max_seqlen, Hk, Hv,
                       dk, dv, total_tokens=None, scale=None, max_tokens=None, workspace=None,
                       stream=None) -> None:
    """GDN over B packed streams of different lengths (cu_seqlens, device int32 [B+1])."""
    B = cu_seqlens.shape[0] - 1
    total = q.shape[0] if total_tokens is None else total_tokens
    scale = 1.0 / math.sqrt(dk) if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_load().la_gdn_prefill_varlen(
        _ptr(h_state_ptrs), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(out),
        _ptr(cu_seqlens), B, total, max_seqlen,
        max_tokens if max_tokens is not None else total, Hk, Hv, dk, dv, _row_stride(q),
        _row_stride(k), _row_stride(v), float(scale), _dtype_code(q), _ptr(workspace), ws_bytes,
        _stream(stream)))


def gdn_prefill_varlen_noalloc(h_state_ptrs, q, k, v, g, beta, out, cu_seqlens, *, max_seqlen,
                               Hk, Hv, dk, dv, total_tokens=None, scale=None, max_tokens=None,
                               stream=None) -> None:
    """gdn_prefill_varlen without a workspace, for callers that cannot allocate device memory:
    the library's fixed scratch (up to 4096 streams per call) is used instead. Calls that
    overlap on the GPU share that scratch and must be ordered; the first call on a device
    should come before any stream capture there. The entry point is compiled for bf16 q, k, v
    and out only: any other dtype is refused here (the C call has no dtype argument)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"gdn_prefill_varlen_noalloc takes bf16 tensors; {name} is {t.dtype}")
    B = cu_seqlens.shape[0] - 1
    total = q.shape[0] if total_tokens is None else total_tokens
    scale = 1.0 / math.sqrt(dk) if scale is None else scale
    _check(_load().la_gdn_prefill_varlen_noalloc(
        _ptr(h_state_ptrs), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(out),
        _ptr(cu_seqlens), B, total, max_seqlen,
        max_tokens if max_tokens is not None else total, Hk, Hv, dk, dv, _row_stride(q),
        _row_stride(k), _row_stride(v), float(scale), _stream(stream)))


def kda_prefill(h_state_ptrs, q, k, v, gate, beta, out, cu_seqlens=None, *, Hk, Hv, dk, dv,
                max_seqlen=None, total_tokens=None, scale=None, pad_fill=0.0, max_tokens=None,
                workspace=None, stream=None) -> None:
    """KDA (per-channel gate [tok][Hv][dk]) over one stream (cu_seqlens None) or B streams."""
    B = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    total = q.shape[0] if total_tokens is None else total_tokens
    max_seqlen = total if max_seqlen is None else max_seqlen
    scale = 1.0 / math.sqrt(dk) if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_load().la_kda_prefill(
        _ptr(h_state_ptrs), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta), _ptr(out),
        _ptr(cu_seqlens), B, total, max_seqlen,
        max_tokens if max_tokens is not None else total, Hk, Hv, dk, dv, _row_stride(q),
        _row_stride(k), _row_stride(v), float(scale), float(pad_fill), _dtype_code(q),
        _ptr(workspace), ws_bytes, _stream(stream)))


def prefill_front(conv_state_ptrs, h_state_ptrs, x, conv_w, gate, beta, out, cu_seqlens=None, *,
                  B=None, Hk, Hv, dk, dv, kda, conv_bias=None, max_seqlen=None,
                  total_tokens=None, l2_eps=1e-6, scale=None, pad_fill=0.0, max_tokens=None,
                  z=None, norm_w=None, norm_eps=1e-6, workspace=None, stream=None) -> None:
    """conv1d + SiLU + q|k L2 + recurrence of one layer in one launch, from the pre-conv rows
    x [tok][2*Hk*dk + Hv*dv]. cu_seqlens None: B equal streams (B defaults to 1). With z (and
    norm_w [dv]) the output store applies the gated RMSNorm o/rms(o) * norm_w * SiLU(z)."""
    if cu_seqlens is not None:
        B = cu_seqlens.shape[0] - 1
    elif B is None:
        B = 1
    total = x.shape[0] if total_tokens is None else total_tokens
    max_seqlen = (total // B if cu_seqlens is None else total) if max_seqlen is None else max_seqlen
    scale = 1.0 / math.sqrt(dk) if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _, K = conv_w.shape
    _check(_load().la_prefill_front(
        _ptr(conv_state_ptrs), _ptr(h_state_ptrs), _ptr(x), _ptr(conv_w), _ptr(conv_bias), K,
        _ptr(gate), _ptr(beta), _ptr(out), _ptr(cu_seqlens), B, total, max_seqlen,
        max_tokens if max_tokens is not None else total, Hk, Hv, dk, dv, _row_stride(x),
        float(l2_eps), float(scale), float(pad_fill), _ptr(z), _ptr(norm_w), float(norm_eps),
        1 if kda else 0, _dtype_code(x), _ptr(workspace), ws_bytes, _stream(stream)))


def decode_workspace_bytes(B, Hk, Hv, dk, dv, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (LA_BF16 if dtype == torch.bfloat16 else LA_F32)
    return int(_load().la_decode_workspace_bytes(B, Hk, Hv, dk, dv, code))


def decode_step(conv_state_ptrs, h_state_ptrs, x, conv_w, gate, beta, out, *, Hk, Hv, dk, dv,
                kda, conv_bias=None, l2_eps=1e-6, scale=None, max_streams=None, workspace=None,
                stream=None) -> None:
    """One decode step: x [B][cd] holds one new token per stream; conv and h states advance
    in place; out [B][Hv][dv]."""
    B = x.shape[0]
    scale = 1.0 / math.sqrt(dk) if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _, K = conv_w.shape
    _check(_load().la_decode_step(
        _ptr(conv_state_ptrs), _ptr(h_state_ptrs), _ptr(x), _ptr(conv_w), _ptr(conv_bias), K,
        _ptr(gate), _ptr(beta), _ptr(out), B, max_streams if max_streams is not None else B, Hk,
        Hv, dk, dv, _row_stride(x), float(l2_eps), float(scale), 1 if kda else 0,
        _dtype_code(x), _ptr(workspace), ws_bytes, _stream(stream)))


def gated_rmsnorm(o, z, w, y=None, *, eps=1e-6, stream=None):
    """y = o / sqrt(mean(o^2) + eps) * w * SiLU(z) per row of the last axis; o, z [t][Hv][dv].
    y defaults to o (in place). Returns y."""
    y = o if y is None else y
    t, Hv, dv = o.shape
    _check(_load().la_gated_rmsnorm(_ptr(o), _ptr(z), _ptr(w), _ptr(y), t, Hv, dv, float(eps),
                                    _dtype_code(o), _stream(stream)))
    return y


def gemm_bf16(a, w, c=None, *, stream=None):
    """C = A W^T (bf16, fp32 accumulation on the tensor cores); a [M][K], w [N][K] (a linear
    layer's [out][in] weight); c [M][N] (allocated when None). Returns c."""
    M, K = a.shape
    N = w.shape[0]
    if c is None:
        c = torch.empty(M, N, dtype=torch.bfloat16, device=a.device)
    _check(_load().la_gemm_bf16(_ptr(a), _ptr(w), _ptr(c), M, N, K, _row_stride(a),
                                _row_stride(w), _row_stride(c), _stream(stream)))
    return c


def rmsnorm_rows(x, w, y=None, *, eps=1e-6, stream=None):
    """y = x / sqrt(mean(x^2) + eps) * w per row (bf16); y defaults to a new tensor."""
    rows, width = x.shape
    if y is None:
        y = torch.empty_like(x)
    _check(_load().la_rmsnorm_rows(_ptr(x), _ptr(w), _ptr(y), rows, width, _row_stride(x),
                                   _row_stride(y), float(eps), _stream(stream)))
    return y


def gate_activations(ab, na, g=None, beta=None, *, stream=None):
    """g = -softplus(ab[:, :na]), beta = sigmoid(ab[:, na:]) in fp32 (new tensors by default)."""
    t, width = ab.shape
    nb = width - na
    if g is None:
        g = torch.empty(t, na, dtype=torch.float32, device=ab.device)
    if beta is None:
        beta = torch.empty(t, nb, dtype=torch.float32, device=ab.device)
    _check(_load().la_gate_activations(_ptr(ab), _row_stride(ab), t, na, nb, _ptr(g), _ptr(beta),
                                       _stream(stream)))
    return g, beta


def prefill_segmented_workspace_bytes(total_tokens, Hv, segments) -> int:
    return int(_load().la_prefill_segmented_workspace_bytes(total_tokens, Hv, segments))


def prefill_segmented(h_state_ptrs, q, k, v, gate, beta, out, *, Hk, Hv, dk, dv, kda, segments,
                      total_tokens=None, scale=None, max_tokens=None, workspace=None,
                      stream=None) -> None:
    """The recurrence of ONE long stream with its tokens cut into `segments` pieces that run
    side by side on the tensor cores, then joined (chunk-parallel scan)."""
    total = q.shape[0] if total_tokens is None else total_tokens
    scale = 1.0 / math.sqrt(dk) if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_load().la_prefill_segmented(
        _ptr(h_state_ptrs), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta), _ptr(out), total,
        max_tokens if max_tokens is not None else total, Hk, Hv, dk, dv, _row_stride(q),
        _row_stride(k), _row_stride(v), float(scale), 1 if kda else 0, int(segments),
        _dtype_code(q), _ptr(workspace), ws_bytes, _stream(stream)))
