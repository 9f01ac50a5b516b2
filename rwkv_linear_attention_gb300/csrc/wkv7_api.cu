// Host side of the C ABI (include/wkv7.h): argument validation, the
// per-device status word, and the launches.  No call allocates memory.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "sm103_ptx.cuh"
#include "wkv7_internal.cuh"

namespace {

// One status word per device, set by kernels with atomicOr and read/cleared
// by wkv7_check_device_status.
__device__ unsigned g_wkv7_device_status = 0u;

constexpr int kMaxDevices = 64;
std::mutex g_status_mutex;
unsigned *g_status_ptr[kMaxDevices] = {};

thread_local char g_last_cuda_error[256] = "";

wkv7_status cuda_fail(cudaError_t e) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return WKV7_ERR_CUDA;
}

// Device address of the status word on the current device (looked up once).
wkv7_status status_word(unsigned **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return WKV7_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_wkv7_device_status);
        if (e != cudaSuccess) return cuda_fail(e);
        g_status_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_status_ptr[dev];
    return WKV7_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte ranges [p, p + n) and [q, q + m) overlap.
bool overlaps(const void *p, size_t n, const void *q, size_t m) {
    if (!p || !q || n == 0 || m == 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + m && b < a + n;
}

// One wait that nothing completes, through the same bounded-wait helper and
// status report as the kernels' mbarrier waits: the device gives up after
// timeout_ns and reports kDevTimeout.
__global__ void wkv7_bounded_wait_probe_kernel(unsigned *status, unsigned long long timeout_ns) {
    __shared__ alignas(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = wkv7::ptx::smem_addr(&bar);
    wkv7::ptx::mbar_init(b, 1);
    wkv7::ptx::fence_mbar_init();
    if (!wkv7::ptx::mbar_wait_bounded(b, 0, 1u << 24, timeout_ns)) wkv7::report(status, wkv7::kDevTimeout);
}

constexpr long long kMaxHeads = 1ll << 30;   // B*H (or num_seqs*H) limit
constexpr long long kMaxTokens = 1ll << 31;  // int32 token indices

}  // namespace

extern "C" {

int wkv7_abi_version(void) { return 100; }

const char *wkv7_last_cuda_error(void) { return g_last_cuda_error; }

const char *wkv7_status_string(wkv7_status s) {
    switch (s) {
        case WKV7_OK: return "ok";
        case WKV7_ERR_INVALID_ARG: return "invalid argument";
        case WKV7_ERR_UNSUPPORTED: return "unsupported (only head size N = 64 is supported)";
        case WKV7_ERR_ALIGNMENT: return "a tensor pointer is not 16-byte aligned";
        case WKV7_ERR_CUDA: return "CUDA error";
        case WKV7_ERR_TIMEOUT: return "a bounded device-side wait expired";
        case WKV7_ERR_WORKSPACE: return "workspace missing or too small";
        case WKV7_ERR_DEVICE_BOUNDS: return "device found an index out of range";
    }
    return "unknown status";
}

wkv7_status wkv7_step_cast(int B, int H, int N, const float *r, const float *w, const float *k,
                           const float *v, const float *kk, const float *a, float *state, void *o,
                           wkv7_dtype o_dtype, cudaStream_t stream) {
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (o_dtype != WKV7_F32 && o_dtype != WKV7_BF16) return WKV7_ERR_UNSUPPORTED;
    if (B < 0 || H <= 0) return WKV7_ERR_INVALID_ARG;
    const long long heads = (long long)B * H;
    if (heads > kMaxHeads) return WKV7_ERR_INVALID_ARG;
    if (heads == 0) return WKV7_OK;
    const void *ptrs[8] = {r, w, k, v, kk, a, state, o};
    for (const void *p : ptrs)
        if (!p) return WKV7_ERR_INVALID_ARG;
    for (const void *p : ptrs)
        if (!aligned16(p)) return WKV7_ERR_ALIGNMENT;
    const size_t vec_bytes = (size_t)heads * N * sizeof(float);
    const size_t o_bytes = (size_t)heads * N * (o_dtype == WKV7_BF16 ? 2 : 4);
    const size_t state_bytes = vec_bytes * N;
    const void *ins[6] = {r, w, k, v, kk, a};
    for (const void *p : ins)
        if (overlaps(state, state_bytes, p, vec_bytes)) return WKV7_ERR_INVALID_ARG;
    if (overlaps(state, state_bytes, o, o_bytes)) return WKV7_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (overlaps(o, o_bytes, ins[i], vec_bytes)) return WKV7_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;
    cudaError_t e = wkv7::launch_step(heads, r, w, k, v, kk, a, state, o, o_dtype, nullptr, status, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_step_state(int B, int H, int N, const float *r, const float *w, const float *k, const float *v,
                            const float *kk, const float *a, void *state, wkv7_dtype state_dtype, void *o,
                            wkv7_dtype o_dtype, cudaStream_t stream) {
    if (state_dtype == WKV7_F32)
        return wkv7_step_cast(B, H, N, r, w, k, v, kk, a, static_cast<float *>(state), o, o_dtype, stream);
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (state_dtype != WKV7_F16 && state_dtype != WKV7_BF16) return WKV7_ERR_UNSUPPORTED;
    if (o_dtype != WKV7_F32 && o_dtype != WKV7_BF16) return WKV7_ERR_UNSUPPORTED;
    if (B < 0 || H <= 0) return WKV7_ERR_INVALID_ARG;
    const long long heads = (long long)B * H;
    if (heads > kMaxHeads) return WKV7_ERR_INVALID_ARG;
    if (heads == 0) return WKV7_OK;
    const void *ptrs[8] = {r, w, k, v, kk, a, state, o};
    for (const void *p : ptrs)
        if (!p) return WKV7_ERR_INVALID_ARG;
    for (const void *p : ptrs)
        if (!aligned16(p)) return WKV7_ERR_ALIGNMENT;
    const size_t vec_bytes = (size_t)heads * N * sizeof(float);
    const size_t o_bytes = (size_t)heads * N * (o_dtype == WKV7_BF16 ? 2 : 4);
    const size_t state_bytes = (size_t)heads * N * N * 2;
    const void *ins[6] = {r, w, k, v, kk, a};
    for (const void *p : ins)
        if (overlaps(state, state_bytes, p, vec_bytes)) return WKV7_ERR_INVALID_ARG;
    if (overlaps(state, state_bytes, o, o_bytes)) return WKV7_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (overlaps(o, o_bytes, ins[i], vec_bytes)) return WKV7_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;
    cudaError_t e = wkv7::launch_step_state16(heads, r, w, k, v, kk, a, state, state_dtype, o, o_dtype, status, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_step(int B, int H, int N, const float *r, const float *w, const float *k,
                      const float *v, const float *kk, const float *a, float *state, float *o,
                      cudaStream_t stream) {
    return wkv7_step_cast(B, H, N, r, w, k, v, kk, a, state, o, WKV7_F32, stream);
}

wkv7_status wkv7_step_tail(int B, int H, int N, const float *r, const float *w, const float *k,
                           const float *v, const float *kk, const float *a, float *state, float *o,
                           const float *r_k, const float *ln_w, const float *ln_b, const float *g,
                           float eps, float *y, cudaStream_t stream) {
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (B < 0 || H <= 0 || !(eps >= 0.f) || !std::isfinite(eps)) return WKV7_ERR_INVALID_ARG;
    const long long heads = (long long)B * H;
    if (heads > kMaxHeads) return WKV7_ERR_INVALID_ARG;
    if (heads == 0) return WKV7_OK;
    const void *ptrs[12] = {r, w, k, v, kk, a, state, r_k, ln_w, ln_b, g, y};
    for (const void *p : ptrs)
        if (!p) return WKV7_ERR_INVALID_ARG;
    for (const void *p : ptrs)
        if (!aligned16(p)) return WKV7_ERR_ALIGNMENT;
    if (o && !aligned16(o)) return WKV7_ERR_ALIGNMENT;
    const size_t vec_bytes = (size_t)heads * N * sizeof(float);
    const size_t state_bytes = vec_bytes * N;
    const size_t par_bytes = (size_t)H * N * sizeof(float);
    const void *ins[9] = {r, w, k, v, kk, a, g, o, y};
    for (const void *p : ins)
        if (overlaps(state, state_bytes, p, vec_bytes)) return WKV7_ERR_INVALID_ARG;
    for (const float *p : {r_k, ln_w, ln_b})
        if (overlaps(state, state_bytes, p, par_bytes)) return WKV7_ERR_INVALID_ARG;
    // the outputs o (when given) and y overlap no input, no parameter and not each other
    for (const void *out : {(const void *)o, (const void *)y}) {
        for (int i = 0; i < 7; ++i)
            if (overlaps(out, vec_bytes, ins[i], vec_bytes)) return WKV7_ERR_INVALID_ARG;
        for (const float *p : {r_k, ln_w, ln_b})
            if (overlaps(out, vec_bytes, p, par_bytes)) return WKV7_ERR_INVALID_ARG;
    }
    if (overlaps(o, vec_bytes, y, vec_bytes)) return WKV7_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;
    const wkv7::TailArgs tail{r_k, ln_w, ln_b, g, y, eps, H};
    cudaError_t e = wkv7::launch_step(heads, r, w, k, v, kk, a, state, o, WKV7_F32, &tail, status, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_verify(int B, int T, int H, int N, const float *r, const float *w, const float *k, const float *v,
                        const float *kk, const float *a, const float *state, float *o, float *states,
                        cudaStream_t stream) {
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (B < 0 || H <= 0 || T < 1 || T > wkv7::verify_max_tokens()) return WKV7_ERR_INVALID_ARG;
    const long long heads = (long long)B * H;
    if (heads * T > kMaxHeads) return WKV7_ERR_INVALID_ARG;
    if (heads == 0) return WKV7_OK;
    const void *ptrs[10] = {r, w, k, v, kk, a, state, o, states, nullptr};
    for (int i = 0; i < 9; ++i)
        if (!ptrs[i]) return WKV7_ERR_INVALID_ARG;
    for (int i = 0; i < 9; ++i)
        if (!aligned16(ptrs[i])) return WKV7_ERR_ALIGNMENT;
    const size_t vec_bytes = (size_t)heads * T * N * sizeof(float);
    const size_t state_bytes = (size_t)heads * N * N * sizeof(float);
    const size_t states_bytes = state_bytes * T;
    const void *ins[6] = {r, w, k, v, kk, a};
    for (const void *p : ins) {
        if (overlaps(o, vec_bytes, p, vec_bytes) || overlaps(states, states_bytes, p, vec_bytes))
            return WKV7_ERR_INVALID_ARG;
    }
    if (overlaps(o, vec_bytes, state, state_bytes) || overlaps(states, states_bytes, state, state_bytes) ||
        overlaps(o, vec_bytes, states, states_bytes))
        return WKV7_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;
    cudaError_t e = wkv7::launch_verify(B, T, H, r, w, k, v, kk, a, state, o, states, status, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_verify_commit(int B, int T, int H, int N, const float *states, const int32_t *accept_len,
                               float *state, cudaStream_t stream) {
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (B < 0 || H <= 0 || T < 1 || T > wkv7::verify_max_tokens()) return WKV7_ERR_INVALID_ARG;
    const long long heads = (long long)B * H;
    if (heads * T > kMaxHeads) return WKV7_ERR_INVALID_ARG;
    if (heads == 0) return WKV7_OK;
    if (!states || !accept_len || !state) return WKV7_ERR_INVALID_ARG;
    if (!aligned16(states) || !aligned16(state)) return WKV7_ERR_ALIGNMENT;
    const size_t state_bytes = (size_t)heads * N * N * sizeof(float);
    if (overlaps(state, state_bytes, states, state_bytes * T) ||
        overlaps(state, state_bytes, accept_len, (size_t)B * sizeof(int32_t)))
        return WKV7_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;
    cudaError_t e = wkv7::launch_verify_commit(B, T, H, states, accept_len, state, status, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_tmix_tail(int n_rows, int H, int N, wkv7_dtype x_dtype, const float *o, const void *r,
                           const void *k, const void *v, const void *g, const float *r_k, const float *ln_w,
                           const float *ln_b, float eps, float *y, cudaStream_t stream) {
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (x_dtype != WKV7_F32 && x_dtype != WKV7_BF16) return WKV7_ERR_UNSUPPORTED;
    if (n_rows < 0 || H <= 0 || !(eps >= 0.f) || !std::isfinite(eps)) return WKV7_ERR_INVALID_ARG;
    if ((long long)n_rows * H > kMaxHeads * 64) return WKV7_ERR_INVALID_ARG;
    if (n_rows == 0) return WKV7_OK;
    const void *ptrs[9] = {o, r, k, v, g, r_k, ln_w, ln_b, y};
    for (const void *p : ptrs)
        if (!p) return WKV7_ERR_INVALID_ARG;
    for (const void *p : ptrs)
        if (!aligned16(p)) return WKV7_ERR_ALIGNMENT;
    const size_t x_elem = x_dtype == WKV7_BF16 ? 2 : 4;
    const size_t elems = (size_t)n_rows * H * N;
    const size_t par_bytes = (size_t)H * N * sizeof(float);
    // y may be o itself (in place) but overlaps nothing else
    if (y != o && overlaps(y, elems * 4, o, elems * 4)) return WKV7_ERR_INVALID_ARG;
    for (const void *p : {r, k, v, g})
        if (overlaps(y, elems * 4, p, elems * x_elem)) return WKV7_ERR_INVALID_ARG;
    for (const float *p : {r_k, ln_w, ln_b})
        if (overlaps(y, elems * 4, p, par_bytes)) return WKV7_ERR_INVALID_ARG;
    const wkv7::TailArgs tail{r_k, ln_w, ln_b, g, y, eps, H};
    cudaError_t e = wkv7::launch_tmix_tail(n_rows, x_dtype, o, r, k, v, tail, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

size_t wkv7_prefill_workspace_size(int num_seqs, int T_total, int H, int N) {
    if (N != wkv7::kN || num_seqs < 0 || T_total < 0 || H <= 0) return 0;
    return wkv7::prefill_workspace_bytes(num_seqs, T_total, H);
}

wkv7_status wkv7_prefill_state(int num_seqs, int T_total, int H, int N, const int32_t *cu_seqlens,
                               const int32_t *cu_seqlens_host, wkv7_dtype x_dtype, const void *r,
                               const float *w, const void *k, const void *v, const void *kk,
                               const void *a, const void *initial_state, void *final_state,
                               wkv7_dtype state_dtype, void *o, wkv7_dtype o_dtype, void *workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (x_dtype != WKV7_F32 && x_dtype != WKV7_BF16 && x_dtype != WKV7_TF32) return WKV7_ERR_UNSUPPORTED;
    if (o_dtype != WKV7_F32 && o_dtype != WKV7_BF16) return WKV7_ERR_UNSUPPORTED;
    if (state_dtype != WKV7_F32 && state_dtype != WKV7_F16 && state_dtype != WKV7_BF16) return WKV7_ERR_UNSUPPORTED;
    if (num_seqs < 0 || T_total < 0 || H <= 0) return WKV7_ERR_INVALID_ARG;
    if ((long long)num_seqs * H > kMaxHeads || (long long)T_total * H * N >= (1ll << 62))
        return WKV7_ERR_INVALID_ARG;
    if ((long long)T_total >= kMaxTokens) return WKV7_ERR_INVALID_ARG;
    if (num_seqs == 0) return T_total == 0 ? WKV7_OK : WKV7_ERR_INVALID_ARG;
    if (!cu_seqlens) return WKV7_ERR_INVALID_ARG;
    if (T_total > 0 && (!r || !w || !k || !v || !kk || !a || !o)) return WKV7_ERR_INVALID_ARG;
    const void *ptrs[11] = {cu_seqlens, r, w, k, v, kk, a, initial_state, final_state, o, nullptr};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return WKV7_ERR_ALIGNMENT;

    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[num_seqs] != T_total)
            return WKV7_ERR_INVALID_ARG;
        for (int b = 0; b < num_seqs; ++b)
            if (cu_seqlens_host[b + 1] < cu_seqlens_host[b]) return WKV7_ERR_INVALID_ARG;
    }

    const size_t x_elem = x_dtype == WKV7_BF16 ? 2 : 4;
    const size_t tok_elems = (size_t)T_total * H * N;
    const size_t state_bytes = (size_t)num_seqs * H * N * N * wkv7::state_elem_bytes(state_dtype);
    const size_t o_bytes = tok_elems * (o_dtype == WKV7_BF16 ? 2 : 4);
    // Outputs must not overlap inputs; final_state may equal initial_state
    // exactly but must not partially overlap it.
    const void *xins[5] = {r, k, v, kk, a};
    for (const void *p : xins) {
        if (overlaps(o, o_bytes, p, tok_elems * x_elem)) return WKV7_ERR_INVALID_ARG;
        if (overlaps(final_state, state_bytes, p, tok_elems * x_elem)) return WKV7_ERR_INVALID_ARG;
    }
    if (overlaps(o, o_bytes, w, tok_elems * 4) || overlaps(final_state, state_bytes, w, tok_elems * 4))
        return WKV7_ERR_INVALID_ARG;
    if (overlaps(o, o_bytes, final_state, state_bytes) || overlaps(o, o_bytes, initial_state, state_bytes))
        return WKV7_ERR_INVALID_ARG;
    if (final_state != initial_state && overlaps(final_state, state_bytes, initial_state, state_bytes))
        return WKV7_ERR_INVALID_ARG;
    if (overlaps(o, o_bytes, cu_seqlens, (size_t)(num_seqs + 1) * 4) ||
        overlaps(final_state, state_bytes, cu_seqlens, (size_t)(num_seqs + 1) * 4))
        return WKV7_ERR_INVALID_ARG;

    // Only the sequence order is required; a larger workspace (up to
    // wkv7_prefill_workspace_size) also enables the tail-split schedule.
    const size_t need = wkv7::prefill_workspace_min_bytes(num_seqs);
    if (need > 0 && (!workspace || workspace_bytes < need)) return WKV7_ERR_WORKSPACE;
    if (!workspace) workspace_bytes = 0;
    if (workspace_bytes > 0) {
        if (!aligned16(workspace)) return WKV7_ERR_ALIGNMENT;
        const void *others[9] = {o, final_state, initial_state, r, w, k, v, kk, a};
        const size_t sizes[9] = {o_bytes, state_bytes, state_bytes, tok_elems * x_elem, tok_elems * 4,
                                 tok_elems * x_elem, tok_elems * x_elem, tok_elems * x_elem, tok_elems * x_elem};
        for (int i = 0; i < 9; ++i)
            if (overlaps(workspace, workspace_bytes, others[i], sizes[i])) return WKV7_ERR_INVALID_ARG;
        if (overlaps(workspace, workspace_bytes, cu_seqlens, (size_t)(num_seqs + 1) * 4)) return WKV7_ERR_INVALID_ARG;
    }

    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;

    wkv7::PrefillArgs args;
    args.num_seqs = num_seqs;
    args.T_total = T_total;
    args.H = H;
    args.cu_seqlens = cu_seqlens;
    args.lens = nullptr;
    args.lens_host = nullptr;
    args.row_stride = 0;
    args.order = nullptr;
    args.cu_seqlens_host = cu_seqlens_host;
    args.x_dtype = x_dtype;
    args.r = r; args.w = w; args.k = k; args.v = v; args.kk = kk; args.a = a;
    args.initial_state = initial_state;
    args.final_state = final_state;
    args.o = o;
    args.o_dtype = o_dtype;
    args.state_dtype = state_dtype;
    args.status = status;
    cudaError_t e = cudaSuccess;
    if (need > 0 && wkv7::prefill_wants_order(args)) {
        int32_t *order = static_cast<int32_t *>(workspace);
        e = wkv7::launch_prefill_order(args, order, stream);
        if (e != cudaSuccess) return cuda_fail(e);
        args.order = order;
    }
    e = wkv7::launch_prefill(args, workspace, workspace_bytes, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_prefill_cast(int num_seqs, int T_total, int H, int N, const int32_t *cu_seqlens,
                              const int32_t *cu_seqlens_host, wkv7_dtype x_dtype, const void *r,
                              const float *w, const void *k, const void *v, const void *kk,
                              const void *a, const float *initial_state, float *final_state,
                              void *o, wkv7_dtype o_dtype, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    return wkv7_prefill_state(num_seqs, T_total, H, N, cu_seqlens, cu_seqlens_host, x_dtype, r, w, k, v, kk, a,
                              initial_state, final_state, WKV7_F32, o, o_dtype, workspace, workspace_bytes, stream);
}

wkv7_status wkv7_prefill_padded(int B, int T_max, int H, int N, const int32_t *lens, const int32_t *lens_host,
                                wkv7_dtype x_dtype, const void *r, const float *w, const void *k, const void *v,
                                const void *kk, const void *a, const float *initial_state, float *final_state,
                                void *o, wkv7_dtype o_dtype, void *workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (x_dtype != WKV7_F32 && x_dtype != WKV7_BF16 && x_dtype != WKV7_TF32) return WKV7_ERR_UNSUPPORTED;
    if (o_dtype != WKV7_F32 && o_dtype != WKV7_BF16) return WKV7_ERR_UNSUPPORTED;
    if (B < 0 || T_max < 0 || H <= 0) return WKV7_ERR_INVALID_ARG;
    if ((long long)B * H > kMaxHeads || (long long)B * T_max >= kMaxTokens ||
        (long long)B * T_max * H * N >= (1ll << 62))
        return WKV7_ERR_INVALID_ARG;
    if (B == 0) return WKV7_OK;
    const int T_total = B * T_max;
    if (!lens) return WKV7_ERR_INVALID_ARG;
    if (T_total > 0 && (!r || !w || !k || !v || !kk || !a || !o)) return WKV7_ERR_INVALID_ARG;
    const void *ptrs[10] = {r, w, k, v, kk, a, initial_state, final_state, o, lens};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return WKV7_ERR_ALIGNMENT;
    if (lens_host)
        for (int b = 0; b < B; ++b)
            if (lens_host[b] < 0 || lens_host[b] > T_max) return WKV7_ERR_INVALID_ARG;
    const size_t x_elem = x_dtype == WKV7_BF16 ? 2 : 4;
    const size_t tok_elems = (size_t)T_total * H * N;
    const size_t state_bytes = (size_t)B * H * N * N * sizeof(float);
    const size_t o_bytes = tok_elems * (o_dtype == WKV7_BF16 ? 2 : 4);
    const void *xins[5] = {r, k, v, kk, a};
    for (const void *p : xins) {
        if (overlaps(o, o_bytes, p, tok_elems * x_elem)) return WKV7_ERR_INVALID_ARG;
        if (overlaps(final_state, state_bytes, p, tok_elems * x_elem)) return WKV7_ERR_INVALID_ARG;
    }
    if (overlaps(o, o_bytes, w, tok_elems * 4) || overlaps(final_state, state_bytes, w, tok_elems * 4))
        return WKV7_ERR_INVALID_ARG;
    if (overlaps(o, o_bytes, final_state, state_bytes) || overlaps(o, o_bytes, initial_state, state_bytes))
        return WKV7_ERR_INVALID_ARG;
    if (final_state != initial_state && overlaps(final_state, state_bytes, initial_state, state_bytes))
        return WKV7_ERR_INVALID_ARG;
    if (overlaps(o, o_bytes, lens, (size_t)B * 4) || overlaps(final_state, state_bytes, lens, (size_t)B * 4))
        return WKV7_ERR_INVALID_ARG;
    const size_t need = wkv7::prefill_workspace_min_bytes(B);
    if (need > 0 && (!workspace || workspace_bytes < need)) return WKV7_ERR_WORKSPACE;
    if (!workspace) workspace_bytes = 0;
    if (workspace_bytes > 0) {
        if (!aligned16(workspace)) return WKV7_ERR_ALIGNMENT;
        const void *others[10] = {o, final_state, initial_state, r, w, k, v, kk, a, lens};
        const size_t sizes[10] = {o_bytes, state_bytes, state_bytes, tok_elems * x_elem, tok_elems * 4,
                                  tok_elems * x_elem, tok_elems * x_elem, tok_elems * x_elem, tok_elems * x_elem,
                                  (size_t)B * 4};
        for (int i = 0; i < 10; ++i)
            if (overlaps(workspace, workspace_bytes, others[i], sizes[i])) return WKV7_ERR_INVALID_ARG;
    }
    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;
    wkv7::PrefillArgs args;
    args.num_seqs = B;
    args.T_total = T_total;
    args.H = H;
    args.cu_seqlens = nullptr;
    args.lens = lens;
    args.lens_host = lens_host;
    args.row_stride = T_max;
    args.order = nullptr;
    args.cu_seqlens_host = nullptr;
    args.x_dtype = x_dtype;
    args.r = r; args.w = w; args.k = k; args.v = v; args.kk = kk; args.a = a;
    args.initial_state = initial_state;
    args.final_state = final_state;
    args.o = o;
    args.o_dtype = o_dtype;
    args.state_dtype = WKV7_F32;
    args.status = status;
    cudaError_t e = cudaSuccess;
    if (need > 0 && wkv7::prefill_wants_order(args)) {
        int32_t *order = static_cast<int32_t *>(workspace);
        e = wkv7::launch_prefill_order(args, order, stream);
        if (e != cudaSuccess) return cuda_fail(e);
        args.order = order;
    }
    e = wkv7::launch_prefill(args, workspace, workspace_bytes, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_prefill(int num_seqs, int T_total, int H, int N, const int32_t *cu_seqlens,
                         const int32_t *cu_seqlens_host, wkv7_dtype x_dtype, const void *r,
                         const float *w, const void *k, const void *v, const void *kk,
                         const void *a, const float *initial_state, float *final_state,
                         float *o, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
    return wkv7_prefill_cast(num_seqs, T_total, H, N, cu_seqlens, cu_seqlens_host, x_dtype, r, w, k, v, kk, a,
                             initial_state, final_state, o, WKV7_F32, workspace, workspace_bytes, stream);
}

size_t wkv7_prefill_backward_workspace_size(int num_seqs, int T_total, int H, int N) {
    if (N != wkv7::kN || num_seqs < 0 || T_total < 0 || H <= 0) return 0;
    if ((long long)num_seqs * H > kMaxHeads || (long long)T_total >= kMaxTokens) return 0;
    return wkv7::prefill_backward_workspace_bytes(num_seqs, T_total, H);
}

wkv7_status wkv7_prefill_backward(int num_seqs, int T_total, int H, int N, const int32_t *cu_seqlens,
                                  const int32_t *cu_seqlens_host, wkv7_dtype x_dtype, const void *r,
                                  const float *w, const void *k, const void *v, const void *kk, const void *a,
                                  const float *initial_state, const float *d_o, const float *d_final_state,
                                  float *dr, float *dw, float *dk, float *dv, float *dkk, float *da,
                                  float *d_initial_state, void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
    if (N != wkv7::kN) return WKV7_ERR_UNSUPPORTED;
    if (x_dtype != WKV7_F32 && x_dtype != WKV7_BF16 && x_dtype != WKV7_TF32) return WKV7_ERR_UNSUPPORTED;
    if (num_seqs < 0 || T_total < 0 || H <= 0) return WKV7_ERR_INVALID_ARG;
    if ((long long)num_seqs * H > kMaxHeads || (long long)T_total >= kMaxTokens) return WKV7_ERR_INVALID_ARG;
    if (H > 65535) return WKV7_ERR_INVALID_ARG;  // grid y
    if (num_seqs == 0) return T_total == 0 ? WKV7_OK : WKV7_ERR_INVALID_ARG;
    if (!cu_seqlens) return WKV7_ERR_INVALID_ARG;
    if (T_total > 0 && (!r || !w || !k || !v || !kk || !a || !d_o || !dr || !dw || !dk || !dv || !dkk || !da))
        return WKV7_ERR_INVALID_ARG;
    const void *ptrs[17] = {cu_seqlens, r, w, k, v, kk, a, initial_state, d_o, d_final_state,
                            dr, dw, dk, dv, dkk, da, d_initial_state};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return WKV7_ERR_ALIGNMENT;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[num_seqs] != T_total) return WKV7_ERR_INVALID_ARG;
        for (int b = 0; b < num_seqs; ++b)
            if (cu_seqlens_host[b + 1] < cu_seqlens_host[b]) return WKV7_ERR_INVALID_ARG;
    }
    const size_t need = wkv7::prefill_backward_workspace_bytes(num_seqs, T_total, H);
    if (!workspace || workspace_bytes < need) return WKV7_ERR_WORKSPACE;
    if (!aligned16(workspace)) return WKV7_ERR_ALIGNMENT;

    // Every written range (the six gradients, d_initial_state, the workspace)
    // must not overlap any other argument.
    const size_t x_elem = x_dtype == WKV7_BF16 ? 2 : 4;
    const size_t tok = (size_t)T_total * H * N;
    const size_t st_bytes = (size_t)num_seqs * H * N * N * sizeof(float);
    const void *outs[8] = {dr, dw, dk, dv, dkk, da, d_initial_state, workspace};
    const size_t out_sizes[8] = {tok * 4, tok * 4, tok * 4, tok * 4, tok * 4, tok * 4, st_bytes, workspace_bytes};
    const void *all[17] = {r, k, v, kk, a, w, d_o, initial_state, d_final_state, cu_seqlens,
                           dr, dw, dk, dv, dkk, da, d_initial_state};
    const size_t all_sizes[17] = {tok * x_elem, tok * x_elem, tok * x_elem, tok * x_elem, tok * x_elem, tok * 4,
                                  tok * 4, st_bytes, st_bytes, (size_t)(num_seqs + 1) * 4,
                                  tok * 4, tok * 4, tok * 4, tok * 4, tok * 4, tok * 4, st_bytes};
    for (int i = 0; i < 8; ++i)
        for (int j = 0; j < 17; ++j) {
            if (j >= 10 && j - 10 == i) continue;  // itself
            if (overlaps(outs[i], out_sizes[i], all[j], all_sizes[j])) return WKV7_ERR_INVALID_ARG;
        }

    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;
    wkv7::BackwardArgs b;
    b.num_seqs = num_seqs;
    b.T_total = T_total;
    b.H = H;
    b.cu_seqlens = cu_seqlens;
    b.x_dtype = x_dtype == WKV7_TF32 ? WKV7_F32 : x_dtype;
    b.r = r; b.w = w; b.k = k; b.v = v; b.kk = kk; b.a = a;
    b.initial_state = initial_state;
    b.d_o = d_o;
    b.d_final_state = d_final_state;
    b.dr = dr; b.dw = dw; b.dk = dk; b.dv = dv; b.dkk = dkk; b.da = da;
    b.d_initial_state = d_initial_state;
    b.status = status;
    cudaError_t e = wkv7::launch_prefill_backward(b, workspace, stream);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_diag_bounded_wait(unsigned timeout_us, cudaStream_t stream) {
    if (timeout_us == 0 || timeout_us > 2000000u) return WKV7_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    wkv7_status st = status_word(&status);
    if (st != WKV7_OK) return st;
    wkv7_bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(status, 1000ull * timeout_us);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e);
}

wkv7_status wkv7_check_device_status(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned host = 0;
    e = cudaMemcpyFromSymbol(&host, g_wkv7_device_status, sizeof(host));
    if (e != cudaSuccess) return cuda_fail(e);
    if (host) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_wkv7_device_status, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (host & wkv7::kDevTimeout) return WKV7_ERR_TIMEOUT;
    if (host & wkv7::kDevBounds) return WKV7_ERR_DEVICE_BOUNDS;
    if (host & (wkv7::kDevBadSeqlens | wkv7::kDevDomain)) return WKV7_ERR_INVALID_ARG;
    return WKV7_OK;
}

}  // extern "C"
