// Decode step of the WKV-7 recurrence: one token for B*H heads, the fp32
// state read and written in place.
//
// Per head (Core AI model zoo note "Recurrent / linear-attention LLMs on
// Core AI", section 1), with S = [K, V]:
//     z = kk^T S ;  S' = diag(exp w) S - (kk .* a) z^T + k v^T ;  o = S'^T r
//
// The step moves 32 KB of state per head (read + write) against 1.8 KB of
// vectors, so it is bound by HBM bandwidth.  Work split: the 64 value columns
// of a head evolve independently given the per-row vectors, so a head is cut
// into four 16-column slices and each slice is one warp's private problem --
// no shared memory and no block-level barrier.  Lane L owns the eight key rows
// 8*(L>>2) .. 8*(L>>2)+7 and the four value columns 4*(L&3) .. +3 of its
// slice, i.e. eight float4 (128-bit) words of state.  Each warp load
// instruction covers eight rows x 64 contiguous bytes.  The two reductions
// over the key rows (kk^T S and S'^T r) are a per-lane sum over eight rows
// followed by three xor-shuffles across the row groups.
#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

constexpr int kWarpsPerBlock = 4;  // one head per 128-thread block
constexpr int kSlices = 4;         // 16-column slices per head

__device__ __forceinline__ float4 ld_state(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ void st_state(float *p, const float4 &x) {
    *reinterpret_cast<float4 *>(p) = x;
}
__device__ __forceinline__ float4 ld_in(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ float comp(const float4 &x, int c) {
    return c == 0 ? x.x : c == 1 ? x.y : c == 2 ? x.z : x.w;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
wkv7_step_kernel(long long n_units, const float *__restrict__ r, const float *__restrict__ w,
                 const float *__restrict__ k, const float *__restrict__ v,
                 const float *__restrict__ kk, const float *__restrict__ a,
                 float *__restrict__ state, float *__restrict__ o) {
    const int lane = threadIdx.x & 31;
    const long long unit = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (unit >= n_units) return;
    const long long head = unit / kSlices;
    const int slice = (int)(unit % kSlices);
    const int rg = lane >> 2;         // row group: rows 8*rg .. 8*rg+7
    const int col = slice * 16 + (lane & 3) * 4;
    const int row0 = rg * 8;

    // State first: the bulk of the bytes, all eight loads in flight at once.
    float *S = state + head * (kN * kN) + (long long)row0 * kN + col;
    float4 s[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) s[m] = ld_state(S + m * kN);

    const long long vb = head * kN + row0;
    const float4 w0 = ld_in(w + vb), w1 = ld_in(w + vb + 4);
    const float4 kk0 = ld_in(kk + vb), kk1 = ld_in(kk + vb + 4);
    const float4 a0 = ld_in(a + vb), a1 = ld_in(a + vb + 4);
    const float4 k0 = ld_in(k + vb), k1 = ld_in(k + vb + 4);
    const float4 r0 = ld_in(r + vb), r1 = ld_in(r + vb + 4);
    const float4 vv = ld_in(v + head * kN + col);

    float kkr[8], kr[8], rr[8], dr[8], cr[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        kkr[m] = comp(kk0, m); kkr[m + 4] = comp(kk1, m);
        kr[m] = comp(k0, m);   kr[m + 4] = comp(k1, m);
        rr[m] = comp(r0, m);   rr[m + 4] = comp(r1, m);
        dr[m] = expf(comp(w0, m)); dr[m + 4] = expf(comp(w1, m));
        cr[m] = comp(kk0, m) * comp(a0, m); cr[m + 4] = comp(kk1, m) * comp(a1, m);
    }

    // z = kk^T S over the old state: eight rows here, 64 rows across lanes.
    float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        z0 = fmaf(kkr[m], s[m].x, z0);
        z1 = fmaf(kkr[m], s[m].y, z1);
        z2 = fmaf(kkr[m], s[m].z, z2);
        z3 = fmaf(kkr[m], s[m].w, z3);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        z0 += __shfl_xor_sync(0xffffffffu, z0, off);
        z1 += __shfl_xor_sync(0xffffffffu, z1, off);
        z2 += __shfl_xor_sync(0xffffffffu, z2, off);
        z3 += __shfl_xor_sync(0xffffffffu, z3, off);
    }

    // S' = diag(exp w) S - (kk .* a) z^T + k v^T, then o = S'^T r.
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float d = dr[m], c = cr[m], kv = kr[m];
        s[m].x = fmaf(d, s[m].x, fmaf(-c, z0, kv * vv.x));
        s[m].y = fmaf(d, s[m].y, fmaf(-c, z1, kv * vv.y));
        s[m].z = fmaf(d, s[m].z, fmaf(-c, z2, kv * vv.z));
        s[m].w = fmaf(d, s[m].w, fmaf(-c, z3, kv * vv.w));
        o0 = fmaf(rr[m], s[m].x, o0);
        o1 = fmaf(rr[m], s[m].y, o1);
        o2 = fmaf(rr[m], s[m].z, o2);
        o3 = fmaf(rr[m], s[m].w, o3);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) st_state(S + m * kN, s[m]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        o0 += __shfl_xor_sync(0xffffffffu, o0, off);
        o1 += __shfl_xor_sync(0xffffffffu, o1, off);
        o2 += __shfl_xor_sync(0xffffffffu, o2, off);
        o3 += __shfl_xor_sync(0xffffffffu, o3, off);
    }
    if (rg == 0) *reinterpret_cast<float4 *>(o + head * kN + col) = make_float4(o0, o1, o2, o3);
}

}  // namespace

cudaError_t launch_step(long long n_heads, const float *r, const float *w, const float *k,
                        const float *v, const float *kk, const float *a, float *state,
                        float *o, cudaStream_t stream) {
    if (n_heads <= 0) return cudaSuccess;
    const long long n_units = n_heads * kSlices;
    const long long blocks = (n_units + kWarpsPerBlock - 1) / kWarpsPerBlock;
    wkv7_step_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(
        n_units, r, w, k, v, kk, a, state, o);
    return cudaGetLastError();
}

}  // namespace wkv7
