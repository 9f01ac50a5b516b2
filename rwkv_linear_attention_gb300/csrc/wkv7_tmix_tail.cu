// The time-mix tail after WKV over packed rows (a prefill's outputs), per (row,
// head) of 64 channels:
//     y = (GroupNorm_head(o) * ln_w + ln_b + (sum_i r_i k_i rk_i) v) * g
// The SwiftRWKV inference page names the parts of this tail (group norm, bonus,
// gate) and runs it over the B*T rows of a prompt with the kernel its decode
// step uses; the RWKV-X page lists rk as a per-head weight.  The group is one
// head, the variance is the mean squared deviation, eps comes from the caller.
//
// One warp per (row, head); lane L owns channels 2L, 2L+1.  The mean, the
// variance (two passes) and the bonus are warp sums by shuffles.  The pass is
// bound by HBM traffic: per (row, head) it reads o (256 B), r, k, v and g (128 B
// each in bf16, 256 B in fp32) and writes y (256 B); the parameters stay in L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float2 load2(const float *p) { return *reinterpret_cast<const float2 *>(p); }
__device__ __forceinline__ float2 load2(const __nv_bfloat16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <typename X>
__global__ void __launch_bounds__(kWarps * 32)
wkv7_tmix_tail_kernel(long long n_units, const float *__restrict__ o, const X *__restrict__ r,
                      const X *__restrict__ k, const X *__restrict__ v, TailArgs t) {
    const long long unit = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (unit >= n_units) return;
    const int lane = threadIdx.x & 31;
    const int hp = static_cast<int>(unit % t.H);
    const long long base = unit * kN + 2 * lane;
    const int pb = hp * kN + 2 * lane;
    const float2 ov = load2(o + base);
    const float2 rv = load2(r + base), kv = load2(k + base), vv = load2(v + base);
    const float2 gv = load2(static_cast<const X *>(t.g) + base);
    const float2 rk = load2(t.rk + pb), lw = load2(t.ln_w + pb), lb = load2(t.ln_b + pb);
    const float mean = warp_sum(ov.x + ov.y) * (1.f / kN);
    const float d0 = ov.x - mean, d1 = ov.y - mean;
    const float var = warp_sum(fmaf(d0, d0, d1 * d1)) * (1.f / kN);
    const float bonus = warp_sum(fmaf(rv.x * kv.x, rk.x, rv.y * kv.y * rk.y));
    const float rstd = rsqrtf(var + t.eps);
    const float y0 = (fmaf(d0 * rstd, lw.x, lb.x) + bonus * vv.x) * gv.x;
    const float y1 = (fmaf(d1 * rstd, lw.y, lb.y) + bonus * vv.y) * gv.y;
    *reinterpret_cast<float2 *>(t.y + base) = make_float2(y0, y1);
}

}  // namespace

cudaError_t launch_tmix_tail(long long n_rows, wkv7_dtype x_dtype, const float *o, const void *r,
                             const void *k, const void *v, const TailArgs &tail, cudaStream_t stream) {
    const long long units = n_rows * tail.H;
    if (units <= 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((units + kWarps - 1) / kWarps);
    if (x_dtype == WKV7_BF16)
        wkv7_tmix_tail_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, stream>>>(
            units, o, static_cast<const __nv_bfloat16 *>(r), static_cast<const __nv_bfloat16 *>(k),
            static_cast<const __nv_bfloat16 *>(v), tail);
    else
        wkv7_tmix_tail_kernel<float><<<grid, kWarps * 32, 0, stream>>>(
            units, o, static_cast<const float *>(r), static_cast<const float *>(k), static_cast<const float *>(v),
            tail);
    return cudaGetLastError();
}

}  // namespace wkv7
