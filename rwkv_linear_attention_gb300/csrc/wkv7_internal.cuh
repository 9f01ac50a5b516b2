// Internal declarations shared by the host API and the kernel translation
// units.  Not part of the C ABI (that is include/wkv7.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "wkv7.h"

namespace wkv7 {

constexpr int kN = 64;  // head size: the only one supported

// Bits of the per-device status word (read by wkv7_check_device_status).
enum : unsigned {
    kDevTimeout = 1u,     // a bounded wait expired
    kDevBounds = 2u,      // an index was out of range
    kDevBadSeqlens = 4u,  // device cu_seqlens malformed
    kDevDomain = 8u,      // an input lies outside a kernel's stated domain (w < kMinLogDecay)
};

// Smallest log-decay the chunked kernels (prefill and its backward) accept.  They
// take a chunk's decay factors relative to its 32nd token, so each scaled operand
// carries a factor within e^{+-32|w|max}; a product of two of them (the removal
// block C^T T Q of the chunk transition, where one channel's growth meets
// another's through T) reaches e^{64|w|max}, which must stay well inside fp32
// (e^{88.7}).  With w >= -1 that is e^{64}.  RWKV-7 models have w in (-0.6066, 0).
constexpr float kMinLogDecay = -1.0f;

__device__ __forceinline__ void report(unsigned *status, unsigned bit) {
    if (status) atomicOr(status, bit);
}

// The time-mix tail after WKV, per (row, head) of N = 64 channels:
//   y = (GroupNorm_head(o) * ln_w + ln_b + (sum_i r_i k_i rk_i) v) * g
struct TailArgs {
    const float *rk;    // [H, 64]
    const float *ln_w;  // [H, 64]
    const float *ln_b;  // [H, 64]
    const void *g;      // [rows, H, 64], the row inputs' type
    float *y;           // [rows, H, 64] fp32
    float eps;
    int H;
};

// Decode: one token for n_heads = B * H heads; o of o_dtype (fp32 or bf16); with
// `tail` the time-mix tail is fused into the epilogue (o fp32, may then be null).
cudaError_t launch_step(long long n_heads, const float *r, const float *w, const float *k,
                        const float *v, const float *kk, const float *a, float *state,
                        void *o, wkv7_dtype o_dtype, const TailArgs *tail, unsigned *status,
                        cudaStream_t stream);

// Decode with the state stored in 16 bits (state_dtype WKV7_F16 or WKV7_BF16): widened
// to fp32 on load, rounded to nearest even on store; o of o_dtype (fp32 or bf16).
cudaError_t launch_step_state16(long long n_heads, const float *r, const float *w, const float *k, const float *v,
                                const float *kk, const float *a, void *state, wkv7_dtype state_dtype, void *o,
                                wkv7_dtype o_dtype, unsigned *status, cudaStream_t stream);

// Multi-token verify (speculative decoding): T tokens per row from a read-only state,
// every position's state kept; and the rollback to each row's accepted length.
int verify_max_tokens();
cudaError_t launch_verify(int B, int T, int H, const float *r, const float *w, const float *k, const float *v,
                          const float *kk, const float *a, const float *state, float *o, float *states,
                          unsigned *status, cudaStream_t stream);
cudaError_t launch_verify_commit(int B, int T, int H, const float *states, const int32_t *accept_len, float *state,
                                 unsigned *status, cudaStream_t stream);

// The time-mix tail over packed rows: o fp32 [n_rows, H, 64]; r, k, v, g of x_dtype.
cudaError_t launch_tmix_tail(long long n_rows, wkv7_dtype x_dtype, const float *o, const void *r,
                             const void *k, const void *v, const TailArgs &tail, cudaStream_t stream);

struct PrefillArgs {
    int num_seqs;
    int T_total;
    int H;
    const int32_t *cu_seqlens;   // device [num_seqs + 1], or nullptr with `lens`
    const int32_t *lens;         // padded layout: device [num_seqs]; sequence b owns tokens
    const int32_t *lens_host;    //   b * row_stride .. b * row_stride + lens[b] - 1 (host copy or nullptr)
    int row_stride;
    const int32_t *order;        // device [num_seqs] schedule (longest first) or nullptr
    const int32_t *cu_seqlens_host;  // host copy of cu_seqlens or nullptr (scheduling only)
    wkv7_dtype x_dtype;
    const void *r;
    const float *w;
    const void *k;
    const void *v;
    const void *kk;
    const void *a;
    const void *initial_state;   // nullable, [num_seqs, H, 64, 64] of state_dtype
    void *final_state;           // nullable, same type
    void *o;                     // [T_total, H, 64] of o_dtype
    wkv7_dtype o_dtype;          // WKV7_F32, or WKV7_BF16 (rounded to nearest even)
    wkv7_dtype state_dtype;      // WKV7_F32, WKV7_F16 or WKV7_BF16 (16-bit: rounded to nearest even)
    unsigned *status;            // device status word
};

// Four consecutive state elements at element index idx of a state array of type dt,
// widened to fp32; and the rounded store (to nearest even for the 16-bit types).
__device__ __forceinline__ float4 load_state4(const void *base, wkv7_dtype dt, long long idx) {
    if (dt == WKV7_F32) return *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + idx);
    const uint2 u = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(base) + idx);
    if (dt == WKV7_BF16)
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                           __uint_as_float(u.y & 0xffff0000u));
    const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ void store_state4(void *base, wkv7_dtype dt, long long idx, float4 v) {
    if (dt == WKV7_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(base) + idx) = v;
        return;
    }
    uint2 u;
    if (dt == WKV7_BF16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        u.x = *reinterpret_cast<const uint32_t *>(&lo);
        u.y = *reinterpret_cast<const uint32_t *>(&hi);
    } else {
        const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
        u.x = *reinterpret_cast<const uint32_t *>(&lo);
        u.y = *reinterpret_cast<const uint32_t *>(&hi);
    }
    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(base) + idx) = u;
}
inline size_t state_elem_bytes(wkv7_dtype dt) { return dt == WKV7_F32 ? 4 : 2; }

// Token range [bos, eos) of sequence b: packed (cu_seqlens) or padded (lens, row_stride).
__device__ __forceinline__ void seq_bounds(const PrefillArgs &p, int b, int &bos, int &eos) {
    if (p.lens) {
        bos = b * p.row_stride;
        eos = bos + p.lens[b];
    } else {
        bos = p.cu_seqlens[b];
        eos = p.cu_seqlens[b + 1];
    }
}
// The same on the host from the host copy (cu_seqlens_host or lens_host); false if absent.
inline bool host_seq_len(const PrefillArgs &p, int b, int &len) {
    if (p.lens) {
        if (!p.lens_host) return false;
        len = p.lens_host[b];
        return true;
    }
    if (!p.cu_seqlens_host) return false;
    len = p.cu_seqlens_host[b + 1] - p.cu_seqlens_host[b];
    return true;
}

// Prefill, token-serial form (one warp per 16-column slice, tokens in order).
cudaError_t launch_prefill_scan(const PrefillArgs &args, cudaStream_t stream);

// Prefill: the chunked tensor-core kernel.
cudaError_t launch_prefill(const PrefillArgs &args, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);
size_t prefill_workspace_bytes(int num_seqs, int T_total, int H);  // for the fastest schedule
size_t prefill_workspace_min_bytes(int num_seqs);                 // required (the sequence order)
// Whether this batch is worth a longest-first schedule, and the kernel that
// writes it (order[rank] = sequence index) into device memory.
bool prefill_wants_order(const PrefillArgs &args);
cudaError_t launch_prefill_order(const PrefillArgs &args, int32_t *order, cudaStream_t stream);

// Backward of the packed prefill (chunked; see wkv7_prefill_backward.cu).
struct BackwardArgs {
    int num_seqs;
    int T_total;
    int H;
    const int32_t *cu_seqlens;  // device [num_seqs + 1]
    wkv7_dtype x_dtype;
    const void *r;
    const float *w;
    const void *k;
    const void *v;
    const void *kk;
    const void *a;
    const float *initial_state;  // nullable
    const float *d_o;            // [T_total, H, 64]
    const float *d_final_state;  // nullable
    float *dr, *dw, *dk, *dv, *dkk, *da;  // [T_total, H, 64]
    float *d_initial_state;               // nullable
    unsigned *status;                     // device status word
};
size_t prefill_backward_workspace_bytes(int num_seqs, int T_total, int H);
cudaError_t launch_prefill_backward(const BackwardArgs &args, void *workspace, cudaStream_t stream);

}  // namespace wkv7
