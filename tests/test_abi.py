"""C-ABI checks that need no GPU: the library loads, exports every symbol include/linattn.h
declares, and refuses bad counts and arguments on the host before any CUDA call.

Refusal rule: "glm5next_kda/prefill.rs" — a call covers 1..=max_tokens tokens and any other
count is refused before a launch (module invariant; the bail! of prefill_with_pad_fill).
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")

A = 0x10000  # a 16-byte-aligned fake address: never dereferenced, calls are refused first


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib(built_lib):
    import linear_attention_chunked_conv1d_gb300 as la
    la._load()
    return la


def test_header_declares_the_pages_calls():
    syms = declared_symbols()
    for name in ["la_conv1d_silu_prefill", "la_conv1d_silu_prefill_varlen", "la_l2norm_heads",
                 "la_gdn_prefill_batched", "la_gdn_prefill_varlen", "la_kda_prefill"]:
        assert name in syms


def test_every_declared_symbol_is_exported(built_lib):
    cdll = ctypes.CDLL(built_lib)
    for name in declared_symbols():
        assert hasattr(cdll, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", built_lib], capture_output=True,
                        text=True).stdout
    for name in declared_symbols():
        assert re.search(rf"\bT {name}$", nm, flags=re.M), name


def test_abi_version(lib):
    assert lib.abi_version() == 1


def _rc_conv(lib, t, max_tokens, **kw):
    args = dict(conv_state=A, x=A, w=A, bias=None, out=A * 2, channels=64, kernel=4,
                x_stride=64, out_stride=64, dtype=1)
    args.update(kw)
    return lib._load().la_conv1d_silu_prefill(
        args["conv_state"], args["x"], args["w"], args["bias"], args["out"], t, max_tokens,
        args["channels"], args["kernel"], args["x_stride"], args["out_stride"], args["dtype"], 0)


def test_conv_refuses_counts(lib):
    assert _rc_conv(lib, 0, 10) == lib.LA_ERR_COUNT
    assert _rc_conv(lib, 11, 10) == lib.LA_ERR_COUNT
    assert _rc_conv(lib, -3, 10) == lib.LA_ERR_COUNT
    assert "max_tokens" in lib.last_error()


def test_conv_refuses_bad_args(lib):
    assert _rc_conv(lib, 5, 10, x=A + 2) == lib.LA_ERR_ARG           # misaligned
    assert _rc_conv(lib, 5, 10, x=None) == lib.LA_ERR_ARG            # null
    assert _rc_conv(lib, 5, 10, channels=60) == lib.LA_ERR_ARG       # not 16 B of bf16
    assert _rc_conv(lib, 5, 10, x_stride=32) == lib.LA_ERR_ARG       # stride < width
    assert _rc_conv(lib, 5, 10, out=A) == lib.LA_ERR_ARG             # aliasing
    assert _rc_conv(lib, 5, 10, dtype=7) == lib.LA_ERR_ARG
    assert _rc_conv(lib, 5, 10, kernel=5) == lib.LA_ERR_UNSUPPORTED
    assert _rc_conv(lib, 5, 10, conv_state=None) == lib.LA_ERR_ARG


def test_l2_refusals(lib):
    f = lib._load().la_l2norm_heads
    assert f(A, 0, 2, 128, 256, 1e-6, 1, 0) == lib.LA_ERR_COUNT
    assert f(A, 4, 2, 96, 256, 1e-6, 1, 0) == lib.LA_ERR_UNSUPPORTED
    assert f(A, 4, 2, 128, 200, 1e-6, 1, 0) == lib.LA_ERR_ARG
    assert f(A + 8, 4, 2, 128, 256, 1e-6, 1, 0) == lib.LA_ERR_ARG


def _rc_gdn_batched(lib, B, T, max_tokens, **kw):
    a = dict(Hk=2, Hv=4, dk=128, dv=128, qs=1024, ks=1024, vs=512, dtype=1, ws=None, wsb=0)
    a.update(kw)
    return lib._load().la_gdn_prefill_batched(A, A, A, A, A, A, A * 2, B, T, max_tokens, a["Hk"],
                                              a["Hv"], a["dk"], a["dv"], a["qs"], a["ks"],
                                              a["vs"], 0.1, a["dtype"], a["ws"], a["wsb"], 0)


def test_gdn_batched_refusals(lib):
    assert _rc_gdn_batched(lib, 2, 0, 100) == lib.LA_ERR_COUNT
    assert _rc_gdn_batched(lib, 0, 5, 100) == lib.LA_ERR_COUNT
    assert _rc_gdn_batched(lib, 4, 30, 100) == lib.LA_ERR_COUNT     # 120 > 100
    assert _rc_gdn_batched(lib, 2, 8, 100, Hv=3) == lib.LA_ERR_ARG   # Hv % Hk
    assert _rc_gdn_batched(lib, 2, 8, 100, dk=96, dv=96) == lib.LA_ERR_UNSUPPORTED
    assert _rc_gdn_batched(lib, 2, 8, 100, dk=128, dv=64) == lib.LA_ERR_UNSUPPORTED
    assert _rc_gdn_batched(lib, 2, 8, 100, qs=100) == lib.LA_ERR_ARG


def test_varlen_and_kda_refusals(lib):
    L = lib._load()
    # total 0 / above max_tokens
    assert L.la_gdn_prefill_varlen(A, A, A, A, A, A, A * 2, A, 3, 0, 1, 10, 1, 1, 64, 64, 64, 64,
                                   64, 1.0, 1, None, 0, 0) == lib.LA_ERR_COUNT
    assert L.la_gdn_prefill_varlen(A, A, A, A, A, A, A * 2, A, 3, 11, 5, 10, 1, 1, 64, 64, 64, 64,
                                   64, 1.0, 1, None, 0, 0) == lib.LA_ERR_COUNT
    # null cu_seqlens
    assert L.la_gdn_prefill_varlen(A, A, A, A, A, A, A * 2, None, 3, 9, 5, 10, 1, 1, 64, 64, 64,
                                   64, 64, 1.0, 1, None, 0, 0) == lib.LA_ERR_ARG
    # max_seqlen beyond total
    assert L.la_gdn_prefill_varlen(A, A, A, A, A, A, A * 2, A, 3, 9, 10, 10, 1, 1, 64, 64, 64,
                                   64, 64, 1.0, 1, None, 0, 0) == lib.LA_ERR_ARG
    # KDA: count refusal, and B != 1 without cu_seqlens
    assert L.la_kda_prefill(A, A, A, A, A, A, A * 2, None, 1, 0, 1, 10, 1, 1, 64, 64, 64, 64, 64,
                            1.0, 0.0, 1, None, 0, 0) == lib.LA_ERR_COUNT
    assert L.la_kda_prefill(A, A, A, A, A, A, A * 2, None, 2, 5, 5, 10, 1, 1, 64, 64, 64, 64, 64,
                            1.0, 0.0, 1, None, 0, 0) == lib.LA_ERR_ARG
    assert "max_tokens" in lib.last_error() or "B == 1" in lib.last_error()


def test_binding_raises_typed_error(lib):
    with pytest.raises(lib.LinAttnError) as ei:
        lib._check(lib.LA_ERR_COUNT)
    assert ei.value.code == lib.LA_ERR_COUNT


def test_workspace_query(lib):
    assert lib.prefill_workspace_bytes(4, 1000, 16, 32, 128, 128, lib.LA_BF16) >= 0


def _rc_front(lib, **kw):
    """la_prefill_front with fake addresses; every case here is refused before any launch."""
    a = dict(cs=A, hs=A, x=A, w=A, bias=None, K=4, g=A, beta=A, out=A * 2, cu=A, B=2, total=40,
             max_seqlen=30, max_tokens=100, Hk=1, Hv=2, dk=128, dv=128, xs=512, eps=1e-6,
             scale=0.1, pad=0.0, z=None, nw=None, neps=1e-6, kda=0, dtype=1, ws=A * 3,
             wsb=1 << 20)
    a.update(kw)
    return lib._load().la_prefill_front(
        a["cs"], a["hs"], a["x"], a["w"], a["bias"], a["K"], a["g"], a["beta"], a["out"],
        a["cu"], a["B"], a["total"], a["max_seqlen"], a["max_tokens"], a["Hk"], a["Hv"], a["dk"],
        a["dv"], a["xs"], a["eps"], a["scale"], a["pad"], a["z"], a["nw"], a["neps"], a["kda"],
        a["dtype"], a["ws"], a["wsb"], 0)


def test_fused_prefill_refusals(lib):
    assert _rc_front(lib, total=0) == lib.LA_ERR_COUNT
    assert _rc_front(lib, total=101) == lib.LA_ERR_COUNT
    assert _rc_front(lib, dtype=0) == lib.LA_ERR_UNSUPPORTED          # fp32: separate calls
    assert _rc_front(lib, dk=64, dv=64) == lib.LA_ERR_UNSUPPORTED
    assert _rc_front(lib, K=5) == lib.LA_ERR_UNSUPPORTED
    assert _rc_front(lib, kda=2) == lib.LA_ERR_ARG
    assert _rc_front(lib, Hv=3, Hk=2) == lib.LA_ERR_ARG               # Hv % Hk
    assert _rc_front(lib, cu=None, total=41) == lib.LA_ERR_ARG        # batched: 41 % 2
    assert _rc_front(lib, max_seqlen=41) == lib.LA_ERR_ARG
    assert _rc_front(lib, cs=None) == lib.LA_ERR_ARG                  # conv state needed (K > 1)
    assert _rc_front(lib, x=A + 4) == lib.LA_ERR_ARG                  # misaligned
    assert _rc_front(lib, xs=500) == lib.LA_ERR_ARG                   # stride < 2 Hk dk + Hv dv
    assert _rc_front(lib, out=A) == lib.LA_ERR_ARG                    # aliases x
    assert _rc_front(lib, eps=-1.0) == lib.LA_ERR_ARG
    assert _rc_front(lib, wsb=16) == lib.LA_ERR_ARG                   # workspace too small
    assert _rc_front(lib, ws=None) == lib.LA_ERR_ARG
    assert "workspace" in lib.last_error()
    assert _rc_front(lib, z=A * 4, nw=None) == lib.LA_ERR_ARG          # gated norm: weight needed
    assert _rc_front(lib, z=A * 4 + 2, nw=A * 5) == lib.LA_ERR_ARG     # misaligned z
    assert _rc_front(lib, z=A * 4, nw=A * 5, neps=-1.0) == lib.LA_ERR_ARG


def test_gated_rmsnorm_refusals(lib):
    f = lib._load().la_gated_rmsnorm
    assert f(A, A * 2, A * 3, A * 4, 0, 2, 128, 1e-6, 1, 0) == lib.LA_ERR_COUNT
    assert f(A, A * 2, A * 3, A * 4, 5, 2, 96, 1e-6, 1, 0) == lib.LA_ERR_UNSUPPORTED
    assert f(A, A * 2, A * 3, A * 4, 5, 0, 128, 1e-6, 1, 0) == lib.LA_ERR_ARG
    assert f(A + 2, A * 2, A * 3, A * 4, 5, 2, 128, 1e-6, 1, 0) == lib.LA_ERR_ARG
    assert f(A, A * 2, None, A * 4, 5, 2, 128, 1e-6, 1, 0) == lib.LA_ERR_ARG
    assert f(A, A * 2, A * 3, A * 2, 5, 2, 128, 1e-6, 1, 0) == lib.LA_ERR_ARG   # y aliases z
    assert f(A, A * 2, A * 3, A * 4, 5, 2, 128, -1.0, 1, 0) == lib.LA_ERR_ARG


def test_workspace_grows_with_conv_reader_counts(lib):
    L = lib._load()
    small = L.la_prefill_workspace_bytes(4, 100, 1, 4, 128, 128, 1)
    big = L.la_prefill_workspace_bytes(4, 100, 64, 64, 128, 128, 1)
    assert big > small and big % 16 == 0 and small % 16 == 0


def _rc_decode(lib, **kw):
    """la_decode_step with fake addresses; every case here is refused before any launch."""
    a = dict(cs=A, hs=A, x=A, w=A, bias=None, K=4, g=A, beta=A, out=A * 2, B=4, maxb=8, Hk=1,
             Hv=2, dk=128, dv=128, xs=512, eps=1e-6, scale=0.1, kda=0, dtype=1, ws=A * 3,
             wsb=1 << 20)
    a.update(kw)
    return lib._load().la_decode_step(
        a["cs"], a["hs"], a["x"], a["w"], a["bias"], a["K"], a["g"], a["beta"], a["out"], a["B"],
        a["maxb"], a["Hk"], a["Hv"], a["dk"], a["dv"], a["xs"], a["eps"], a["scale"], a["kda"],
        a["dtype"], a["ws"], a["wsb"], 0)


def test_decode_refusals(lib):
    assert _rc_decode(lib, B=0) == lib.LA_ERR_COUNT
    assert _rc_decode(lib, B=9) == lib.LA_ERR_COUNT
    assert _rc_decode(lib, dk=96, dv=96) == lib.LA_ERR_UNSUPPORTED
    assert _rc_decode(lib, K=0) == lib.LA_ERR_UNSUPPORTED
    assert _rc_decode(lib, Hk=2, Hv=3) == lib.LA_ERR_ARG
    assert _rc_decode(lib, xs=500) == lib.LA_ERR_ARG
    assert _rc_decode(lib, x=A + 2) == lib.LA_ERR_ARG
    assert _rc_decode(lib, hs=None) == lib.LA_ERR_ARG
    assert _rc_decode(lib, wsb=100) == lib.LA_ERR_ARG
    assert _rc_decode(lib, kda=3) == lib.LA_ERR_ARG


def test_decode_workspace_size(lib):
    L = lib._load()
    # one bf16 conv-output row per stream, rounded up to 16 bytes
    assert L.la_decode_workspace_bytes(3, 1, 2, 128, 128, 1) == 3 * 512 * 2
    assert L.la_decode_workspace_bytes(3, 1, 1, 64, 64, 0) == 3 * 192 * 4
    assert L.la_decode_workspace_bytes(0, 1, 1, 64, 64, 0) == 0


def test_gemm_refusals(lib):
    f = lib._load().la_gemm_bf16
    B = A * 16
    assert f(A, B, A * 64, 0, 8, 8, 8, 8, 8, 0) == lib.LA_ERR_COUNT
    assert f(A, B, A * 64, 8, 8, 0, 8, 8, 8, 0) == lib.LA_ERR_COUNT
    assert f(A + 2, B, A * 64, 8, 8, 8, 8, 8, 8, 0) == lib.LA_ERR_ARG       # misaligned
    assert f(A, B, A * 64, 8, 8, 16, 8, 16, 8, 0) == lib.LA_ERR_ARG         # lda < K
    assert f(A, B, A * 64, 8, 8, 12, 12, 16, 8, 0) == lib.LA_ERR_ARG        # lda not 16 B
    assert f(A, B, A * 64, 8, 16, 8, 8, 8, 8, 0) == lib.LA_ERR_ARG          # ldc < N
    assert f(A, B, A + 64, 8, 8, 8, 8, 8, 8, 0) == lib.LA_ERR_ARG           # c overlaps a


def test_phase1_elementwise_refusals(lib):
    L = lib._load()
    assert L.la_rmsnorm_rows(A, A * 2, A * 3, 0, 64, 64, 64, 1e-6, 0) == lib.LA_ERR_COUNT
    assert L.la_rmsnorm_rows(A, A * 2, A * 3, 4, 60, 64, 64, 1e-6, 0) == lib.LA_ERR_UNSUPPORTED
    assert L.la_rmsnorm_rows(A, A * 2, A * 3, 4, 8200, 8200, 8200, 1e-6, 0) == lib.LA_ERR_UNSUPPORTED
    assert L.la_rmsnorm_rows(A + 4, A * 2, A * 3, 4, 64, 64, 64, 1e-6, 0) == lib.LA_ERR_ARG
    assert L.la_rmsnorm_rows(A, A * 2, A * 3, 4, 64, 60, 64, 1e-6, 0) == lib.LA_ERR_ARG
    assert L.la_gate_activations(A, 8, 0, 4, 4, A * 2, A * 3, 0) == lib.LA_ERR_COUNT
    assert L.la_gate_activations(A, 7, 5, 4, 4, A * 2, A * 3, 0) == lib.LA_ERR_ARG
    assert L.la_gate_activations(A, 8, 5, 4, 4, None, A * 3, 0) == lib.LA_ERR_ARG


def test_segmented_refusals(lib):
    L = lib._load()
    args = lambda **kw: dict(dict(total=100, maxt=200, Hk=1, Hv=2, dk=128, dv=128, kda=0, S=2,
                                  dtype=1, ws=A * 64, wsb=1 << 30), **kw)  # noqa: E731

    def rc(**kw):
        a = args(**kw)
        return L.la_prefill_segmented(A, A, A, A, A, A, A * 2, a["total"], a["maxt"], a["Hk"],
                                      a["Hv"], a["dk"], a["dv"], 256, 256, 256, 0.1, a["kda"],
                                      a["S"], a["dtype"], a["ws"], a["wsb"], 0)
    assert rc(total=0) == lib.LA_ERR_COUNT
    assert rc(total=300) == lib.LA_ERR_COUNT
    assert rc(S=0) == lib.LA_ERR_ARG and rc(S=9) == lib.LA_ERR_ARG
    assert rc(dtype=0) == lib.LA_ERR_UNSUPPORTED
    assert rc(dk=64, dv=64) == lib.LA_ERR_UNSUPPORTED
    assert rc(wsb=100) == lib.LA_ERR_ARG
    assert L.la_prefill_segmented_workspace_bytes(4096, 32, 2) > 32 * 128 * 128 * 4 * 3


# ---------------------------------------------------------------- host-side fault injection
@pytest.fixture
def inject(monkeypatch):
    """Sets LA_FAULT_INJECT for one test (the library reads it at every call)."""
    def set_(mode):
        if mode is None:
            monkeypatch.delenv("LA_FAULT_INJECT", raising=False)
        else:
            monkeypatch.setenv("LA_FAULT_INJECT", mode)
    yield set_
    monkeypatch.delenv("LA_FAULT_INJECT", raising=False)


def _valid_calls(lib):
    """One call per launching entry point with arguments that pass every host check (fake,
    aligned addresses: with a fault injected the call returns before any CUDA call)."""
    L = lib._load()
    ws = 1 << 20
    return {
        "conv": lambda: _rc_conv(lib, 5, 10),
        "l2": lambda: L.la_l2norm_heads(A, 4, 2, 128, 256, 1e-6, 1, 0),
        "gdn_batched": lambda: _rc_gdn_batched(lib, 2, 8, 100, ws=A * 64, wsb=ws),
        "gdn_varlen_noalloc": lambda: L.la_gdn_prefill_varlen_noalloc(
            A, A, A, A, A, A, A * 2, A, 3, 9, 5, 10, 1, 1, 128, 128, 128, 128, 128, 1.0, 0),
        "decode": lambda: _rc_decode(lib),
        "gemm": lambda: L.la_gemm_bf16(A, A * 16, A * 64, 8, 8, 8, 8, 8, 8, 0),
        "rmsnorm_rows": lambda: L.la_rmsnorm_rows(A, A * 2, A * 3, 4, 64, 64, 64, 1e-6, 0),
        "gated_rmsnorm": lambda: L.la_gated_rmsnorm(A, A * 2, A * 3, A * 4, 4, 2, 128, 1e-6, 1, 0),
    }


def test_injected_launch_failure_is_reported_before_any_launch(lib, inject):
    inject("launch")
    for name, call in _valid_calls(lib).items():
        assert call() == lib.LA_ERR_CUDA, name
        assert "injected launch failure" in lib.last_error(), (name, lib.last_error())
    # host checks still come first: a refused count is reported as such
    assert _rc_conv(lib, 0, 10) == lib.LA_ERR_COUNT


def test_injected_alloc_failure_is_reported(lib, inject):
    inject("alloc")
    calls = _valid_calls(lib)
    for name in ("conv", "gdn_batched", "gdn_varlen_noalloc", "decode", "gemm"):
        assert calls[name]() == lib.LA_ERR_CUDA, name
        assert "injected allocation failure" in lib.last_error(), (name, lib.last_error())
    assert lib._load().la_device_status(0) == -1  # the status word cannot be had either


def test_unknown_injection_value_is_ignored(lib, inject):
    inject("sometimes")
    assert _rc_conv(lib, 0, 10) == lib.LA_ERR_COUNT
    assert "injected" not in lib.last_error()


def test_noalloc_binding_refuses_non_bf16(lib):
    """The no-allocation call has no dtype argument (it is compiled for bf16): the binding
    refuses any other dtype instead of letting the kernel read fp32 data as bf16."""
    import torch
    T, d = 4, 128
    q = torch.zeros(T, d, dtype=torch.float32)
    bf = torch.zeros(T, d, dtype=torch.bfloat16)
    g = torch.zeros(T, 1)
    cu = torch.tensor([0, T], dtype=torch.int32)
    ptrs = torch.zeros(1, dtype=torch.int64)
    for bad in ("q", "k", "v", "out"):
        t = {n: bf for n in ("q", "k", "v")}
        t["out"] = bf.view(T, 1, d)
        t[bad] = q if bad != "out" else q.view(T, 1, d)
        with pytest.raises(TypeError, match=bad):
            lib.gdn_prefill_varlen_noalloc(ptrs, t["q"], t["k"], t["v"], g, g, t["out"], cu,
                                           max_seqlen=T, Hk=1, Hv=1, dk=d, dv=d)
