// wkv7_prefill_noalloc: the packed varlen prefill for callers that cannot
// hand the library a device workspace.
//
// Some callers cannot allocate device memory at the time they run the
// prefill: a serving engine whose memory planner reserves the whole device up
// front so that request handling never allocates (an allocation mid-request
// is slow and may fail), code that records work during CUDA stream capture,
// where cudaMalloc is not permitted, and host programs that only receive
// pointers to buffers someone else owns.  This entry point takes the same
// inputs and outputs as wkv7_prefill and keeps its scratch -- the
// longest-first order of the sequences -- in a fixed array in device memory
// that this library reserves once, when it is loaded.
#include <cstdint>
#include <mutex>

#include "wkv7_internal.cuh"

namespace {

// Scratch shared by every call on a device: room for the schedule of up to
// WKV7_NOALLOC_MAX_SEQS sequences.  Every GPU that loads the library holds
// these bytes until the process exits.  Each call writes all the entries it
// reads before reading them, so nothing needs clearing between calls.
static __device__ __align__(256) int32_t g_prefill_noalloc_scratch[WKV7_NOALLOC_MAX_SEQS];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in; the address a kernel may use
// comes from cudaGetSymbolAddress, looked up once per device with that device
// current.
wkv7_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WKV7_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return WKV7_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_noalloc_scratch) != cudaSuccess || !p) return WKV7_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return WKV7_OK;
}

}  // namespace

extern "C" wkv7_status wkv7_prefill_noalloc(int num_seqs, int T_total, int H, int N,
                                            const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                            wkv7_dtype x_dtype, const void *r, const float *w,
                                            const void *k, const void *v, const void *kk, const void *a,
                                            const float *initial_state, float *final_state, float *o,
                                            cudaStream_t stream) {
    if (num_seqs > WKV7_NOALLOC_MAX_SEQS) return WKV7_ERR_WORKSPACE;
    const size_t need = N == wkv7::kN ? wkv7::prefill_workspace_min_bytes(num_seqs) : 0;
    if (need > sizeof(g_prefill_noalloc_scratch)) return WKV7_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const wkv7_status st = scratch_address(&scratch);
        if (st != WKV7_OK) return st;
    }
    return wkv7_prefill(num_seqs, T_total, H, N, cu_seqlens, cu_seqlens_host, x_dtype, r, w, k, v, kk, a,
                        initial_state, final_state, o, scratch, need > 0 ? sizeof(g_prefill_noalloc_scratch) : 0,
                        stream);
}
