// C ABI of linattn: host-side validation (every check before any launch) and dispatch.
//
// Error convention follows the pages: "glm5next_kda/prefill.rs" refuses a token count of 0 or
// above the workspace's max_tokens before any launch (module invariant and the bail! at the top
// of prefill_with_pad_fill); "split_prefill.rs" returns an error from calls a layer cannot run
// (prefill_gdn_full_batched's default) — here LA_ERR_UNSUPPORTED for dims outside the compiled
// instances.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return LA_OK;
}

// Per-device status word raised by kernels (LA_DEV_*), read and cleared by la_device_status.
__device__ int g_dev_status;

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices];
std::once_flag g_status_once[kMaxDevices];

// Host-side fault injection for tests: LA_FAULT_INJECT=launch makes every call that passed
// its checks return LA_ERR_CUDA instead of launching; LA_FAULT_INJECT=alloc makes the lookup
// of the library's device arrays fail. Read at every call, so a test can switch it on and off.
enum Inject { INJECT_NONE = 0, INJECT_LAUNCH = 1, INJECT_ALLOC = 2 };

Inject fault_inject() {
    const char *v = getenv("LA_FAULT_INJECT");
    if (!v) return INJECT_NONE;
    if (!strcmp(v, "launch")) return INJECT_LAUNCH;
    if (!strcmp(v, "alloc")) return INJECT_ALLOC;
    return INJECT_NONE;
}

int *status_ptr() {
    if (fault_inject() == INJECT_ALLOC) return nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(g_status_once[dev], [dev] {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dev_status) == cudaSuccess) g_status_ptr[dev] = (int *)p;
    });
    return g_status_ptr[dev];
}

// The status word of the current device, or LA_ERR_CUDA when its address cannot be had. Every
// launching call takes it right before its launch, so an injected launch failure is reported
// here already (before any CUDA call).
int get_status(int **out) {
    *out = nullptr;
    if (fault_inject() == INJECT_LAUNCH)
        return fail(LA_ERR_CUDA, "injected launch failure (LA_FAULT_INJECT=launch)");
    *out = status_ptr();
    if (!*out)
        return fail(LA_ERR_CUDA, fault_inject() == INJECT_ALLOC
                                     ? "injected allocation failure (LA_FAULT_INJECT=alloc)"
                                     : "the device status word could not be looked up");
    return LA_OK;
}

// Limit of the bounded waits inside the tensor-core kernels: 2 s, or LA_WAIT_LIMIT_NS (a test
// knob that lets a wait run out on purpose; read at every call), never below 1 ms: the kernels'
// block-wide error checks rely on a wait running at least that long before it gives up.
uint64_t wait_limit_ns() {
    constexpr uint64_t kMin = 1000000ull;
    const char *v = getenv("LA_WAIT_LIMIT_NS");
    if (v && *v) {
        char *end = nullptr;
        const unsigned long long n = strtoull(v, &end, 10);
        if (end && *end == '\0' && n > 0) return n < kMin ? kMin : (uint64_t)n;
    }
    return 2000000000ull;
}

cudaStream_t as_stream(uint64_t s) { return reinterpret_cast<cudaStream_t>(static_cast<uintptr_t>(s)); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int vec_elems(int dtype) { return dtype == LA_BF16 ? 8 : 4; }

int check_dtype(int dtype) {
    if (dtype != LA_F32 && dtype != LA_BF16)
        return fail(LA_ERR_ARG, "dtype %d is neither LA_F32 (0) nor LA_BF16 (1)", dtype);
    return LA_OK;
}

int check_act_ptr(const void *p, const char *name, bool nullable = false) {
    if (!p) return nullable ? LA_OK : fail(LA_ERR_ARG, "%s is NULL", name);
    if (!aligned16(p)) return fail(LA_ERR_ARG, "%s is not 16-byte aligned", name);
    return LA_OK;
}

int check_stride(int64_t stride, int64_t width, int dtype, const char *name) {
    if (stride < width)
        return fail(LA_ERR_ARG, "%s (%lld) is smaller than the row width (%lld)", name,
                    (long long)stride, (long long)width);
    if (stride % vec_elems(dtype))
        return fail(LA_ERR_ARG, "%s (%lld) is not a multiple of 16 bytes", name, (long long)stride);
    return LA_OK;
}

// Runs a launch (a callable returning cudaError_t) unless a launch failure is injected.
template <class F>
int launch_result(F &&launch, const char *what) {
    if (fault_inject() == INJECT_LAUNCH)
        return fail(LA_ERR_CUDA, "%s: injected launch failure (LA_FAULT_INJECT=launch)", what);
    const cudaError_t e = launch();
    if (e != cudaSuccess) return fail(LA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

#define LA_TRY(expr)              \
    do {                          \
        int _rc = (expr);         \
        if (_rc != LA_OK) return _rc; \
    } while (0)

int conv_common(const void *x, const void *w, const void *bias, const void *out, int channels,
                int kernel, int64_t x_stride, int64_t out_stride, int dtype) {
    LA_TRY(check_dtype(dtype));
    if (kernel < 1 || kernel > 4)
        return fail(LA_ERR_UNSUPPORTED, "conv kernel %d outside the compiled 1..4", kernel);
    if (channels <= 0) return fail(LA_ERR_ARG, "channels must be positive (got %d)", channels);
    if (channels % vec_elems(dtype))
        return fail(LA_ERR_ARG, "channels (%d) is not a multiple of 16 bytes", channels);
    LA_TRY(check_act_ptr(x, "x"));
    LA_TRY(check_act_ptr(out, "out"));
    LA_TRY(check_act_ptr(bias, "bias", true));
    if (!w) return fail(LA_ERR_ARG, "w is NULL");
    LA_TRY(check_stride(x_stride, channels, dtype, "x_stride"));
    LA_TRY(check_stride(out_stride, channels, dtype, "out_stride"));
    if (x == out) return fail(LA_ERR_ARG, "out may not alias x");
    return LA_OK;
}

// Shared checks of the three recurrence calls.
int rec_common(const uint64_t *h_state_ptrs, const void *q, const void *k, const void *v,
               const float *g, const float *beta, const void *out, int B, int Hk, int Hv,
               int dk, int dv, int64_t qs, int64_t ks, int64_t vs, int dtype,
               const void *workspace, size_t workspace_bytes, size_t need) {
    LA_TRY(check_dtype(dtype));
    if (B < 1) return fail(LA_ERR_ARG, "B must be >= 1 (got %d)", B);
    if (Hk < 1 || Hv < 1) return fail(LA_ERR_ARG, "Hk and Hv must be >= 1 (got %d, %d)", Hk, Hv);
    if (Hv % Hk) return fail(LA_ERR_ARG, "Hv (%d) is not a multiple of Hk (%d)", Hv, Hk);
    if ((dk != 64 && dk != 128) || dv != dk)
        return fail(LA_ERR_UNSUPPORTED, "head dims dk=%d dv=%d: compiled for dk = dv in {64, 128}",
                    dk, dv);
    if (!h_state_ptrs) return fail(LA_ERR_ARG, "h_state_ptrs is NULL");
    LA_TRY(check_act_ptr(q, "q"));
    LA_TRY(check_act_ptr(k, "k"));
    LA_TRY(check_act_ptr(v, "v"));
    LA_TRY(check_act_ptr(out, "out"));
    if (!g) return fail(LA_ERR_ARG, "g is NULL");
    if (!beta) return fail(LA_ERR_ARG, "beta is NULL");
    LA_TRY(check_stride(qs, (int64_t)Hk * dk, dtype, "q_stride"));
    LA_TRY(check_stride(ks, (int64_t)Hk * dk, dtype, "k_stride"));
    LA_TRY(check_stride(vs, (int64_t)Hv * dv, dtype, "v_stride"));
    if (workspace_bytes < need)
        return fail(LA_ERR_ARG, "workspace of %zu bytes is below the %zu required", workspace_bytes,
                    need);
    if (need && (!workspace || !aligned16(workspace)))
        return fail(LA_ERR_ARG, "workspace is NULL or not 16-byte aligned");
    return LA_OK;
}

bool uses_tensor_cores(int dtype, int dk, int dv) {
    la::RecArgs a{};
    a.dtype = dtype; a.dk = dk; a.dv = dv;
    return la::chunk_tc_supported(a);
}

// Test knob LA_DEBUG_STALL=1: the tensor-core kernels make one wait on a barrier that nothing
// completes, which runs out after the wait limit (read at every call).
int debug_stall() {
    const char *v = getenv("LA_DEBUG_STALL");
    return v && !strcmp(v, "1") ? 1 : 0;
}

int run_recurrence(la::RecArgs &a, cudaStream_t st) {
    LA_TRY(get_status(&a.status));
    a.wait_ns = wait_limit_ns();
    a.debug_stall = debug_stall();
    if (la::chunk_tc_supported(a))
        return launch_result([&] { return la::launch_chunk_tc(a, st); }, "chunked recurrence (tcgen05) launch");
    return launch_result([&] { return la::launch_chunk_simt(a, st); }, "chunked recurrence launch");
}

}  // namespace

extern "C" {

int la_abi_version(void) { return LA_ABI_VERSION; }

const char *la_last_error(void) { return g_err; }

int la_device_status(uint64_t stream) {
    int *p = status_ptr();
    if (!p) return -1;
    int h = 0;
    cudaStream_t st = as_stream(stream);
    if (cudaMemcpyAsync(&h, p, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return -1;
    if (cudaMemsetAsync(p, 0, sizeof(int), st) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    return h;
}

int la_conv1d_silu_prefill(void *conv_state, const void *x, const void *w, const void *bias,
                           void *out, int t, int max_tokens, int channels, int kernel,
                           int64_t x_stride, int64_t out_stride, int dtype, uint64_t stream) {
    if (t <= 0 || t > max_tokens)
        return fail(LA_ERR_COUNT, "conv1d of %d tokens does not fit max_tokens %d", t, max_tokens);
    LA_TRY(conv_common(x, w, bias, out, channels, kernel, x_stride, out_stride, dtype));
    if (kernel > 1) LA_TRY(check_act_ptr(conv_state, "conv_state"));
    la::ConvArgs a{};
    a.single_state = conv_state;
    a.x = x; a.w = w; a.bias = bias; a.out = out;
    a.cu = nullptr; a.B = 1; a.total = t; a.channels = channels; a.kernel = kernel;
    a.x_stride = x_stride; a.out_stride = out_stride; a.dtype = dtype;
    LA_TRY(get_status(&a.status));
    return launch_result([&] { return la::launch_conv1d_silu(a, as_stream(stream)); }, "conv1d_silu launch");
}

int la_conv1d_silu_prefill_varlen(const uint64_t *conv_state_ptrs, const void *x, const void *w,
                                  const void *bias, void *out, const int32_t *cu_seqlens, int B,
                                  int total_tokens, int max_tokens, int channels, int kernel,
                                  int64_t x_stride, int64_t out_stride, int dtype,
                                  uint64_t stream) {
    if (total_tokens <= 0 || total_tokens > max_tokens)
        return fail(LA_ERR_COUNT, "conv1d of %d tokens does not fit max_tokens %d", total_tokens,
                    max_tokens);
    LA_TRY(conv_common(x, w, bias, out, channels, kernel, x_stride, out_stride, dtype));
    if (B < 1) return fail(LA_ERR_ARG, "B must be >= 1 (got %d)", B);
    if (!cu_seqlens) return fail(LA_ERR_ARG, "cu_seqlens is NULL");
    if (kernel > 1 && !conv_state_ptrs) return fail(LA_ERR_ARG, "conv_state_ptrs is NULL");
    la::ConvArgs a{};
    a.state_ptrs = conv_state_ptrs;
    a.x = x; a.w = w; a.bias = bias; a.out = out;
    a.cu = cu_seqlens; a.B = B; a.total = total_tokens; a.channels = channels; a.kernel = kernel;
    a.x_stride = x_stride; a.out_stride = out_stride; a.dtype = dtype;
    LA_TRY(get_status(&a.status));
    return launch_result([&] { return la::launch_conv1d_silu(a, as_stream(stream)); }, "conv1d_silu launch");
}

int la_conv1d_silu_l2_prefill(const uint64_t *conv_state_ptrs, const void *x, const void *w,
                              const void *bias, void *out, const int32_t *cu_seqlens, int B,
                              int total_tokens, int max_tokens, int channels, int kernel,
                              int l2_heads, int head_dim, float eps, int64_t x_stride,
                              int64_t out_stride, int dtype, uint64_t stream) {
    if (total_tokens <= 0 || total_tokens > max_tokens)
        return fail(LA_ERR_COUNT, "conv1d of %d tokens does not fit max_tokens %d", total_tokens,
                    max_tokens);
    LA_TRY(conv_common(x, w, bias, out, channels, kernel, x_stride, out_stride, dtype));
    if (B < 1) return fail(LA_ERR_ARG, "B must be >= 1 (got %d)", B);
    if (!cu_seqlens && B != 1) return fail(LA_ERR_ARG, "cu_seqlens NULL requires B == 1");
    if (kernel > 1 && !conv_state_ptrs) return fail(LA_ERR_ARG, "conv_state_ptrs is NULL");
    if (head_dim != 64 && head_dim != 128)
        return fail(LA_ERR_UNSUPPORTED, "head_dim %d: compiled for 64 and 128", head_dim);
    if (l2_heads < 0 || (int64_t)l2_heads * head_dim > channels)
        return fail(LA_ERR_ARG, "l2_heads * head_dim (%d x %d) exceeds channels (%d)", l2_heads,
                    head_dim, channels);
    if (!(eps >= 0.f)) return fail(LA_ERR_ARG, "eps must be >= 0");
    la::ConvArgs a{};
    a.state_ptrs = conv_state_ptrs;
    a.x = x; a.w = w; a.bias = bias; a.out = out;
    a.cu = cu_seqlens; a.B = B; a.total = total_tokens; a.channels = channels; a.kernel = kernel;
    a.x_stride = x_stride; a.out_stride = out_stride; a.dtype = dtype;
    a.l2_heads = l2_heads; a.head_dim = head_dim; a.eps = eps;
    LA_TRY(get_status(&a.status));
    return launch_result([&] { return la::launch_conv1d_silu(a, as_stream(stream)); }, "conv1d_silu_l2 launch");
}

int la_l2norm_heads(void *x, int t, int n_heads, int head_dim, int64_t row_stride, float eps,
                    int dtype, uint64_t stream) {
    if (t <= 0) return fail(LA_ERR_COUNT, "l2norm of %d tokens", t);
    LA_TRY(check_dtype(dtype));
    if (head_dim != 64 && head_dim != 128)
        return fail(LA_ERR_UNSUPPORTED, "head_dim %d: compiled for 64 and 128", head_dim);
    if (n_heads < 1) return fail(LA_ERR_ARG, "n_heads must be >= 1 (got %d)", n_heads);
    LA_TRY(check_act_ptr(x, "x"));
    LA_TRY(check_stride(row_stride, (int64_t)n_heads * head_dim, dtype, "row_stride"));
    if (!(eps >= 0.f)) return fail(LA_ERR_ARG, "eps must be >= 0");
    la::L2Args a{x, t, n_heads, head_dim, row_stride, eps, dtype};
    return launch_result([&] { return la::launch_l2norm_heads(a, as_stream(stream)); }, "l2norm launch");
}

size_t la_prefill_workspace_bytes(int B, int total_tokens, int Hk, int Hv, int dk, int dv,
                                  int dtype) {
    (void)total_tokens; (void)Hk; (void)Hv;
    if (B < 1) return 0;
    if (Hk < 0) Hk = 0;
    return uses_tensor_cores(dtype, dk, dv) ? la::chunk_tc_workspace_bytes(B, Hk) : 0;
}

int la_gdn_prefill_batched(const uint64_t *h_state_ptrs, const void *q, const void *k,
                           const void *v, const float *g, const float *beta, void *out, int B,
                           int T, int max_tokens, int Hk, int Hv, int dk, int dv,
                           int64_t q_stride, int64_t k_stride, int64_t v_stride, float scale,
                           int dtype, void *workspace, size_t workspace_bytes, uint64_t stream) {
    if (B < 1 || T < 1 || (int64_t)B * T > max_tokens)
        return fail(LA_ERR_COUNT, "batched prefill of %d x %d tokens does not fit max_tokens %d",
                    B, T, max_tokens);
    const int total = B * T;
    size_t need = la_prefill_workspace_bytes(B, total, Hk, Hv, dk, dv, dtype);
    LA_TRY(rec_common(h_state_ptrs, q, k, v, g, beta, out, B, Hk, Hv, dk, dv, q_stride, k_stride,
                      v_stride, dtype, workspace, workspace_bytes, need));
    la::RecArgs a{};
    a.h_ptrs = h_state_ptrs; a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out;
    a.cu = nullptr; a.B = B; a.T_each = T; a.total = total; a.max_seqlen = T;
    a.Hk = Hk; a.Hv = Hv; a.dk = dk; a.dv = dv;
    a.q_stride = q_stride; a.k_stride = k_stride; a.v_stride = v_stride;
    a.scale = scale; a.pad_fill = 0.f; a.dtype = dtype; a.kda = false;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    return run_recurrence(a, as_stream(stream));
}

int la_gdn_prefill_varlen(const uint64_t *h_state_ptrs, const void *q, const void *k,
                          const void *v, const float *g, const float *beta, void *out,
                          const int32_t *cu_seqlens, int B, int total_tokens, int max_seqlen,
                          int max_tokens, int Hk, int Hv, int dk, int dv, int64_t q_stride,
                          int64_t k_stride, int64_t v_stride, float scale, int dtype,
                          void *workspace, size_t workspace_bytes, uint64_t stream) {
    if (total_tokens <= 0 || total_tokens > max_tokens)
        return fail(LA_ERR_COUNT, "varlen prefill of %d tokens does not fit max_tokens %d",
                    total_tokens, max_tokens);
    if (!cu_seqlens) return fail(LA_ERR_ARG, "cu_seqlens is NULL");
    if (max_seqlen < 1 || max_seqlen > total_tokens)
        return fail(LA_ERR_ARG, "max_seqlen %d outside 1..total_tokens (%d)", max_seqlen,
                    total_tokens);
    size_t need = la_prefill_workspace_bytes(B, total_tokens, Hk, Hv, dk, dv, dtype);
    LA_TRY(rec_common(h_state_ptrs, q, k, v, g, beta, out, B, Hk, Hv, dk, dv, q_stride, k_stride,
                      v_stride, dtype, workspace, workspace_bytes, need));
    la::RecArgs a{};
    a.h_ptrs = h_state_ptrs; a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out;
    a.cu = cu_seqlens; a.B = B; a.T_each = 0; a.total = total_tokens; a.max_seqlen = max_seqlen;
    a.Hk = Hk; a.Hv = Hv; a.dk = dk; a.dv = dv;
    a.q_stride = q_stride; a.k_stride = k_stride; a.v_stride = v_stride;
    a.scale = scale; a.pad_fill = 0.f; a.dtype = dtype; a.kda = false;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    return run_recurrence(a, as_stream(stream));
}

int la_gdn_prefill_varlen_noalloc(const uint64_t *h_state_ptrs, const void *q, const void *k,
                                  const void *v, const float *g, const float *beta, void *out,
                                  const int32_t *cu_seqlens, int B, int total_tokens,
                                  int max_seqlen, int max_tokens, int Hk, int Hv, int dk, int dv,
                                  int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                  float scale, uint64_t stream) {
    if (total_tokens <= 0 || total_tokens > max_tokens)
        return fail(LA_ERR_COUNT, "varlen prefill of %d tokens does not fit max_tokens %d",
                    total_tokens, max_tokens);
    if (!cu_seqlens) return fail(LA_ERR_ARG, "cu_seqlens is NULL");
    if (max_seqlen < 1 || max_seqlen > total_tokens)
        return fail(LA_ERR_ARG, "max_seqlen %d outside 1..total_tokens (%d)", max_seqlen,
                    total_tokens);
    if (!uses_tensor_cores(LA_BF16, dk, dv))
        return fail(LA_ERR_UNSUPPORTED, "the no-allocation call covers bf16 with dk = dv = 128");
    const int max_streams = la::chunk_tc_static_scratch_max_streams();
    if (B > max_streams)
        return fail(LA_ERR_UNSUPPORTED,
                    "%d streams exceed the %d the library's fixed scratch holds; use "
                    "la_gdn_prefill_varlen with a caller workspace", B, max_streams);
    LA_TRY(rec_common(h_state_ptrs, q, k, v, g, beta, out, B, Hk, Hv, dk, dv, q_stride, k_stride,
                      v_stride, LA_BF16, nullptr, 0, 0));
    if (fault_inject() == INJECT_LAUNCH)
        return fail(LA_ERR_CUDA, "injected launch failure (LA_FAULT_INJECT=launch)");
    if (fault_inject() == INJECT_ALLOC)
        return fail(LA_ERR_CUDA, "looking up the fixed scratch: injected allocation failure "
                                 "(LA_FAULT_INJECT=alloc)");
    void *scratch = nullptr;
    size_t scratch_bytes = 0;
    cudaError_t e = la::chunk_tc_static_scratch(&scratch, &scratch_bytes);
    if (e != cudaSuccess)
        return fail(LA_ERR_CUDA, "looking up the fixed scratch: %s", cudaGetErrorString(e));
    la::RecArgs a{};
    a.h_ptrs = h_state_ptrs; a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out;
    a.cu = cu_seqlens; a.B = B; a.T_each = 0; a.total = total_tokens; a.max_seqlen = max_seqlen;
    a.Hk = Hk; a.Hv = Hv; a.dk = dk; a.dv = dv;
    a.q_stride = q_stride; a.k_stride = k_stride; a.v_stride = v_stride;
    a.scale = scale; a.pad_fill = 0.f; a.dtype = LA_BF16; a.kda = false;
    a.workspace = scratch; a.workspace_bytes = scratch_bytes;
    return run_recurrence(a, as_stream(stream));
}

int la_kda_prefill(const uint64_t *h_state_ptrs, const void *q, const void *k, const void *v,
                   const float *gate, const float *beta, void *out, const int32_t *cu_seqlens,
                   int B, int total_tokens, int max_seqlen, int max_tokens, int Hk, int Hv,
                   int dk, int dv, int64_t q_stride, int64_t k_stride, int64_t v_stride,
                   float scale, float pad_fill, int dtype, void *workspace,
                   size_t workspace_bytes, uint64_t stream) {
    if (total_tokens <= 0 || total_tokens > max_tokens)
        return fail(LA_ERR_COUNT, "prefill of %d tokens does not fit a workspace built for %d",
                    total_tokens, max_tokens);
    if (!cu_seqlens) {
        if (B != 1) return fail(LA_ERR_ARG, "cu_seqlens NULL requires B == 1 (got %d)", B);
        max_seqlen = total_tokens;
    } else if (max_seqlen < 1 || max_seqlen > total_tokens) {
        return fail(LA_ERR_ARG, "max_seqlen %d outside 1..total_tokens (%d)", max_seqlen,
                    total_tokens);
    }
    size_t need = la_prefill_workspace_bytes(B, total_tokens, Hk, Hv, dk, dv, dtype);
    LA_TRY(rec_common(h_state_ptrs, q, k, v, gate, beta, out, B, Hk, Hv, dk, dv, q_stride,
                      k_stride, v_stride, dtype, workspace, workspace_bytes, need));
    la::RecArgs a{};
    a.h_ptrs = h_state_ptrs; a.q = q; a.k = k; a.v = v; a.g = gate; a.beta = beta; a.out = out;
    a.cu = cu_seqlens; a.B = B; a.T_each = cu_seqlens ? 0 : total_tokens; a.total = total_tokens;
    a.max_seqlen = max_seqlen;
    a.Hk = Hk; a.Hv = Hv; a.dk = dk; a.dv = dv;
    a.q_stride = q_stride; a.k_stride = k_stride; a.v_stride = v_stride;
    a.scale = scale; a.pad_fill = pad_fill; a.dtype = dtype; a.kda = true;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    return run_recurrence(a, as_stream(stream));
}

int la_prefill_front(const uint64_t *conv_state_ptrs, const uint64_t *h_state_ptrs,
                     const void *x, const void *conv_w, const void *conv_bias, int conv_kernel,
                     const float *g, const float *beta, void *out, const int32_t *cu_seqlens,
                     int B, int total_tokens, int max_seqlen, int max_tokens, int Hk, int Hv,
                     int dk, int dv, int64_t x_stride, float l2_eps, float scale, float pad_fill,
                     const void *z, const void *norm_w, float norm_eps, int kda, int dtype,
                     void *workspace, size_t workspace_bytes, uint64_t stream) {
    if (total_tokens <= 0 || total_tokens > max_tokens)
        return fail(LA_ERR_COUNT, "prefill of %d tokens does not fit max_tokens %d", total_tokens,
                    max_tokens);
    LA_TRY(check_dtype(dtype));
    if (kda != 0 && kda != 1) return fail(LA_ERR_ARG, "kda must be 0 (GDN) or 1 (KDA)");
    if (B < 1) return fail(LA_ERR_ARG, "B must be >= 1 (got %d)", B);
    if (Hk < 1 || Hv < 1) return fail(LA_ERR_ARG, "Hk and Hv must be >= 1 (got %d, %d)", Hk, Hv);
    if (Hv % Hk) return fail(LA_ERR_ARG, "Hv (%d) is not a multiple of Hk (%d)", Hv, Hk);
    if (!uses_tensor_cores(dtype, dk, dv))
        return fail(LA_ERR_UNSUPPORTED,
                    "the fused prefill covers bf16 with dk = dv = 128; use the separate calls");
    if (conv_kernel < 1 || conv_kernel > 4)
        return fail(LA_ERR_UNSUPPORTED, "conv kernel %d outside the compiled 1..4", conv_kernel);
    int T_each = 0;
    if (!cu_seqlens) {
        if (total_tokens % B)
            return fail(LA_ERR_ARG, "cu_seqlens NULL: total_tokens (%d) is not a multiple of B (%d)",
                        total_tokens, B);
        T_each = total_tokens / B;
        max_seqlen = T_each;
    } else if (max_seqlen < 1 || max_seqlen > total_tokens) {
        return fail(LA_ERR_ARG, "max_seqlen %d outside 1..total_tokens (%d)", max_seqlen,
                    total_tokens);
    }
    const int64_t cd = (int64_t)(2 * Hk) * dk + (int64_t)Hv * dv;
    if (!h_state_ptrs) return fail(LA_ERR_ARG, "h_state_ptrs is NULL");
    if (conv_kernel > 1 && !conv_state_ptrs) return fail(LA_ERR_ARG, "conv_state_ptrs is NULL");
    LA_TRY(check_act_ptr(x, "x"));
    LA_TRY(check_act_ptr(out, "out"));
    LA_TRY(check_act_ptr(conv_bias, "conv_bias", true));
    if (!conv_w) return fail(LA_ERR_ARG, "conv_w is NULL");
    if (!g) return fail(LA_ERR_ARG, "g is NULL");
    if (!beta) return fail(LA_ERR_ARG, "beta is NULL");
    LA_TRY(check_stride(x_stride, cd, dtype, "x_stride"));
    if (x == out) return fail(LA_ERR_ARG, "out may not alias x");
    if (!(l2_eps >= 0.f)) return fail(LA_ERR_ARG, "l2_eps must be >= 0");
    if (z) {
        LA_TRY(check_act_ptr(z, "z"));
        LA_TRY(check_act_ptr(norm_w, "norm_w"));
        if (!(norm_eps >= 0.f)) return fail(LA_ERR_ARG, "norm_eps must be >= 0");
        if (z == out) return fail(LA_ERR_ARG, "out may not alias z");
    }
    const size_t need = la_prefill_workspace_bytes(B, total_tokens, Hk, Hv, dk, dv, dtype);
    if (workspace_bytes < need)
        return fail(LA_ERR_ARG, "workspace of %zu bytes is below the %zu required", workspace_bytes,
                    need);
    if (!workspace || !aligned16(workspace))
        return fail(LA_ERR_ARG, "workspace is NULL or not 16-byte aligned");
    la::RecArgs a{};
    a.h_ptrs = h_state_ptrs; a.g = g; a.beta = beta; a.out = out;
    a.cu = cu_seqlens; a.B = B; a.T_each = T_each; a.total = total_tokens;
    a.max_seqlen = max_seqlen;
    a.Hk = Hk; a.Hv = Hv; a.dk = dk; a.dv = dv;
    a.scale = scale; a.pad_fill = pad_fill; a.dtype = dtype; a.kda = kda == 1;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.front = true;
    a.x = x; a.conv_w = conv_w; a.conv_bias = conv_bias; a.conv_state_ptrs = conv_state_ptrs;
    a.x_stride = x_stride; a.conv_k = conv_kernel; a.l2_eps = l2_eps;
    a.z = z; a.norm_w = z ? norm_w : nullptr; a.norm_eps = norm_eps;
    LA_TRY(get_status(&a.status));
    a.wait_ns = wait_limit_ns();
    a.debug_stall = debug_stall();
    return launch_result([&] { return la::launch_chunk_tc(a, as_stream(stream)); }, "fused prefill (tcgen05) launch");
}

int la_gated_rmsnorm(const void *o, const void *z, const void *w, void *y, int t, int Hv, int dv,
                     float eps, int dtype, uint64_t stream) {
    if (t <= 0) return fail(LA_ERR_COUNT, "gated rmsnorm of %d tokens", t);
    LA_TRY(check_dtype(dtype));
    if (dv != 64 && dv != 128)
        return fail(LA_ERR_UNSUPPORTED, "dv %d: compiled for 64 and 128", dv);
    if (Hv < 1) return fail(LA_ERR_ARG, "Hv must be >= 1 (got %d)", Hv);
    LA_TRY(check_act_ptr(o, "o"));
    LA_TRY(check_act_ptr(z, "z"));
    LA_TRY(check_act_ptr(w, "w"));
    LA_TRY(check_act_ptr(y, "y"));
    if (!(eps >= 0.f)) return fail(LA_ERR_ARG, "eps must be >= 0");
    if (y == z) return fail(LA_ERR_ARG, "y may not alias z");
    la::GatedNormArgs a{o, z, w, y, t, Hv, dv, eps, dtype};
    return launch_result([&] { return la::launch_gated_rmsnorm(a, as_stream(stream)); }, "gated rmsnorm launch");
}

size_t la_decode_workspace_bytes(int B, int Hk, int Hv, int dk, int dv, int dtype) {
    if (B < 1 || Hk < 1 || Hv < 1 || dk < 1 || dv < 1) return 0;
    const size_t cd = (size_t)(2 * Hk) * dk + (size_t)Hv * dv;
    const size_t row = (cd * (dtype == LA_BF16 ? 2 : 4) + 15) / 16 * 16;
    return (size_t)B * row;
}

int la_decode_step(const uint64_t *conv_state_ptrs, const uint64_t *h_state_ptrs,
                   const void *x, const void *conv_w, const void *conv_bias, int conv_kernel,
                   const float *g, const float *beta, void *out, int B, int max_streams, int Hk,
                   int Hv, int dk, int dv, int64_t x_stride, float l2_eps, float scale, int kda,
                   int dtype, void *workspace, size_t workspace_bytes, uint64_t stream) {
    if (B < 1 || B > max_streams)
        return fail(LA_ERR_COUNT, "decode step of %d streams does not fit max_streams %d", B,
                    max_streams);
    LA_TRY(check_dtype(dtype));
    if (kda != 0 && kda != 1) return fail(LA_ERR_ARG, "kda must be 0 (GDN) or 1 (KDA)");
    if (Hk < 1 || Hv < 1) return fail(LA_ERR_ARG, "Hk and Hv must be >= 1 (got %d, %d)", Hk, Hv);
    if (Hv % Hk) return fail(LA_ERR_ARG, "Hv (%d) is not a multiple of Hk (%d)", Hv, Hk);
    if ((dk != 64 && dk != 128) || dv != dk)
        return fail(LA_ERR_UNSUPPORTED, "head dims dk=%d dv=%d: compiled for dk = dv in {64, 128}",
                    dk, dv);
    if (conv_kernel < 1 || conv_kernel > 4)
        return fail(LA_ERR_UNSUPPORTED, "conv kernel %d outside the compiled 1..4", conv_kernel);
    const int64_t cd = (int64_t)(2 * Hk) * dk + (int64_t)Hv * dv;
    if (!h_state_ptrs) return fail(LA_ERR_ARG, "h_state_ptrs is NULL");
    if (conv_kernel > 1 && !conv_state_ptrs) return fail(LA_ERR_ARG, "conv_state_ptrs is NULL");
    LA_TRY(check_act_ptr(x, "x"));
    LA_TRY(check_act_ptr(out, "out"));
    LA_TRY(check_act_ptr(conv_bias, "conv_bias", true));
    if (!conv_w) return fail(LA_ERR_ARG, "conv_w is NULL");
    if (!g) return fail(LA_ERR_ARG, "g is NULL");
    if (!beta) return fail(LA_ERR_ARG, "beta is NULL");
    LA_TRY(check_stride(x_stride, cd, dtype, "x_stride"));
    if (x == out) return fail(LA_ERR_ARG, "out may not alias x");
    if (!(l2_eps >= 0.f)) return fail(LA_ERR_ARG, "l2_eps must be >= 0");
    const size_t need = la_decode_workspace_bytes(B, Hk, Hv, dk, dv, dtype);
    if (workspace_bytes < need)
        return fail(LA_ERR_ARG, "workspace of %zu bytes is below the %zu required", workspace_bytes,
                    need);
    if (!workspace || !aligned16(workspace))
        return fail(LA_ERR_ARG, "workspace is NULL or not 16-byte aligned");
    const int64_t row = (int64_t)(need / (size_t)B) / (dtype == LA_BF16 ? 2 : 4);  // elements
    int *status = nullptr;
    LA_TRY(get_status(&status));
    la::ConvArgs c{};
    c.state_ptrs = conv_state_ptrs;
    c.x = x; c.w = conv_w; c.bias = conv_bias; c.out = workspace;
    c.cu = nullptr; c.B = B; c.total = B; c.channels = (int)cd; c.kernel = conv_kernel;
    c.x_stride = x_stride; c.out_stride = row; c.dtype = dtype;
    c.l2_heads = 2 * Hk; c.head_dim = dk; c.eps = l2_eps;
    c.status = status;
    c.one_per_stream = true;
    cudaStream_t st = as_stream(stream);
    LA_TRY(launch_result([&] { return la::launch_conv1d_silu(c, st); }, "decode front end launch"));
    la::DecArgs d{};
    d.h_ptrs = h_state_ptrs; d.qkv = workspace; d.qkv_stride = row;
    d.g = g; d.beta = beta; d.out = out;
    d.B = B; d.Hk = Hk; d.Hv = Hv; d.d = dk; d.scale = scale; d.dtype = dtype; d.kda = kda == 1;
    return launch_result([&] { return la::launch_decode_recurrence(d, st); }, "decode recurrence launch");
}

int la_gemm_bf16(const void *a, const void *w, void *c, int M, int N, int K, int64_t lda,
                 int64_t ldw, int64_t ldc, uint64_t stream) {
    if (M < 1 || N < 1 || K < 1)
        return fail(LA_ERR_COUNT, "gemm of %d x %d x %d", M, N, K);
    LA_TRY(check_act_ptr(a, "a"));
    LA_TRY(check_act_ptr(w, "w"));
    LA_TRY(check_act_ptr(c, "c"));
    LA_TRY(check_stride(lda, K, LA_BF16, "lda"));
    LA_TRY(check_stride(ldw, K, LA_BF16, "ldw"));
    LA_TRY(check_stride(ldc, N, LA_BF16, "ldc"));
    const char *cb = static_cast<const char *>(c), *ce = cb + ((int64_t)(M - 1) * ldc + N) * 2;
    auto overlaps = [&](const void *p, int64_t rows, int64_t ld, int64_t cols) {
        const char *pb = static_cast<const char *>(p), *pe = pb + ((rows - 1) * ld + cols) * 2;
        return pb < ce && cb < pe;
    };
    if (overlaps(a, M, lda, K) || overlaps(w, N, ldw, K))
        return fail(LA_ERR_ARG, "c may not overlap a or w");
    int *status = nullptr;
    LA_TRY(get_status(&status));
    la::GemmArgs g{a, w, c, M, N, K, lda, ldw, ldc, status, wait_limit_ns(), debug_stall()};
    return launch_result([&] { return la::launch_gemm_bf16(g, as_stream(stream)); }, "gemm (tcgen05) launch");
}

int la_rmsnorm_rows(const void *x, const void *w, void *y, int rows, int width, int64_t ldx,
                    int64_t ldy, float eps, uint64_t stream) {
    if (rows < 1) return fail(LA_ERR_COUNT, "rmsnorm of %d rows", rows);
    if (width < 8 || width % 8 || width > la::rmsnorm_rows_max_width())
        return fail(LA_ERR_UNSUPPORTED, "width %d: a multiple of 8 up to %d", width,
                    la::rmsnorm_rows_max_width());
    LA_TRY(check_act_ptr(x, "x"));
    LA_TRY(check_act_ptr(w, "w"));
    LA_TRY(check_act_ptr(y, "y"));
    LA_TRY(check_stride(ldx, width, LA_BF16, "ldx"));
    LA_TRY(check_stride(ldy, width, LA_BF16, "ldy"));
    if (!(eps >= 0.f)) return fail(LA_ERR_ARG, "eps must be >= 0");
    la::RowNormArgs a{x, w, y, rows, width, ldx, ldy, eps};
    return launch_result([&] { return la::launch_rmsnorm_rows(a, as_stream(stream)); }, "rmsnorm launch");
}

int la_gate_activations(const void *ab, int64_t ld, int t, int na, int nb, float *g,
                        float *beta, uint64_t stream) {
    if (t < 1) return fail(LA_ERR_COUNT, "gate activations of %d rows", t);
    if (na < 1 || nb < 1) return fail(LA_ERR_ARG, "na and nb must be >= 1 (got %d, %d)", na, nb);
    if (!ab || !g || !beta) return fail(LA_ERR_ARG, "ab, g and beta must not be NULL");
    if (ld < (int64_t)na + nb) return fail(LA_ERR_ARG, "ld (%lld) is below na + nb", (long long)ld);
    la::GateArgs a{ab, ld, t, na, nb, g, beta};
    return launch_result([&] { return la::launch_gate_activations(a, as_stream(stream)); }, "gate activations launch");
}

size_t la_prefill_segmented_workspace_bytes(int total_tokens, int Hv, int segments) {
    if (total_tokens < 1 || Hv < 1) return 0;
    return la::segmented_workspace_bytes(total_tokens, Hv, segments);
}

int la_prefill_segmented(const uint64_t *h_state_ptrs, const void *q, const void *k,
                         const void *v, const float *g, const float *beta, void *out,
                         int total_tokens, int max_tokens, int Hk, int Hv, int dk, int dv,
                         int64_t q_stride, int64_t k_stride, int64_t v_stride, float scale,
                         int kda, int segments, int dtype, void *workspace,
                         size_t workspace_bytes, uint64_t stream) {
    if (total_tokens <= 0 || total_tokens > max_tokens)
        return fail(LA_ERR_COUNT, "prefill of %d tokens does not fit max_tokens %d", total_tokens,
                    max_tokens);
    if (kda != 0 && kda != 1) return fail(LA_ERR_ARG, "kda must be 0 (GDN) or 1 (KDA)");
    if (segments < 1 || segments > la::kMaxSegments)
        return fail(LA_ERR_ARG, "segments %d outside 1..%d", segments, la::kMaxSegments);
    LA_TRY(check_dtype(dtype));
    if (!uses_tensor_cores(dtype, dk, dv))
        return fail(LA_ERR_UNSUPPORTED, "the segmented scan covers bf16 with dk = dv = 128");
    const size_t need = la_prefill_segmented_workspace_bytes(total_tokens, Hv, segments);
    LA_TRY(rec_common(h_state_ptrs, q, k, v, g, beta, out, 1, Hk, Hv, dk, dv, q_stride, k_stride,
                      v_stride, dtype, workspace, workspace_bytes, need));
    la::RecArgs a{};
    a.h_ptrs = h_state_ptrs; a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out;
    a.cu = nullptr; a.B = 1; a.T_each = total_tokens; a.total = total_tokens;
    a.max_seqlen = total_tokens;
    a.Hk = Hk; a.Hv = Hv; a.dk = dk; a.dv = dv;
    a.q_stride = q_stride; a.k_stride = k_stride; a.v_stride = v_stride;
    a.scale = scale; a.pad_fill = 0.f; a.dtype = dtype; a.kda = kda == 1;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    LA_TRY(get_status(&a.status));
    a.wait_ns = wait_limit_ns();
    return launch_result([&] { return la::launch_segmented(a, segments, as_stream(stream)); }, "segmented scan launch");
}

}  // extern "C"
