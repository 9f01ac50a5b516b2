// Token-serial prefill of the WKV-7 recurrence over packed varlen sequences.
//
// Each (sequence, head) pair runs the per-token update of the Core AI model
// zoo note ("Recurrent / linear-attention LLMs on Core AI", section 1) in
// token order, with the state held in registers for the whole sequence:
// the same warp/lane split as the decode step (a head's 64 value columns cut
// into four 16-column slices, one warp per slice, eight key rows x four
// columns per lane), so each warp reads its inputs once per token and writes
// the state only at the end.  Inputs of token t+1 are loaded while token t is
// computed.
#include <cuda_bf16.h>

#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

constexpr int kWarpsPerBlock = 4;

// Eight consecutive channels as fp32.
template <typename X>
struct In8;
template <>
struct In8<float> {
    float4 lo, hi;
    __device__ __forceinline__ void load(const float *p) {
        lo = __ldg(reinterpret_cast<const float4 *>(p));
        hi = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void unpack(float (&f)[8]) const {
        f[0] = lo.x; f[1] = lo.y; f[2] = lo.z; f[3] = lo.w;
        f[4] = hi.x; f[5] = hi.y; f[6] = hi.z; f[7] = hi.w;
    }
};
template <>
struct In8<__nv_bfloat16> {
    uint4 raw;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
        raw = __ldg(reinterpret_cast<const uint4 *>(p));
    }
    __device__ __forceinline__ void unpack(float (&f)[8]) const {
        const unsigned u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(u[i] << 16);
            f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    }
};

// Four consecutive channels as fp32.
__device__ __forceinline__ void load4(const float *p, float (&f)[4]) {
    const float4 x = __ldg(reinterpret_cast<const float4 *>(p));
    f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&f)[4]) {
    const uint2 x = __ldg(reinterpret_cast<const uint2 *>(p));
    f[0] = __uint_as_float(x.x << 16); f[1] = __uint_as_float(x.x & 0xffff0000u);
    f[2] = __uint_as_float(x.y << 16); f[3] = __uint_as_float(x.y & 0xffff0000u);
}

template <typename X>
struct TokenIn {
    In8<X> r, k, kk, a;
    In8<float> w;
    float v[4];
    __device__ __forceinline__ void load(const X *rp, const float *wp, const X *kp, const X *vp,
                                         const X *kkp, const X *ap, long long row_off,
                                         long long col_off) {
        r.load(rp + row_off);
        w.load(wp + row_off);
        k.load(kp + row_off);
        kk.load(kkp + row_off);
        a.load(ap + row_off);
        load4(vp + col_off, v);
    }
};

template <typename X>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
wkv7_prefill_scan_kernel(PrefillArgs p) {
    const int lane = threadIdx.x & 31;
    const int slice = threadIdx.x >> 5;
    const int H = p.H;
    const long long pair = blockIdx.x;
    const int seq_rank = (int)(pair / H);
    const int h = (int)(pair % H);
    const int b = p.order ? p.order[seq_rank] : seq_rank;
    if (b < 0 || b >= p.num_seqs) {
        if (threadIdx.x == 0) report(p.status, kDevBounds);
        return;
    }
    int bos, eos;
    seq_bounds(p, b, bos, eos);
    if (bos < 0 || eos < bos || eos > p.T_total || (p.lens && eos - bos > p.row_stride)) {
        if (threadIdx.x == 0) report(p.status, kDevBadSeqlens);
        return;
    }

    const int rg = lane >> 2;
    const int row0 = rg * 8;
    const int col = slice * 16 + (lane & 3) * 4;
    const long long slot = ((long long)b * H + h) * (kN * kN) + (long long)row0 * kN + col;

    float4 s[8];
    if (p.initial_state) {
#pragma unroll
        for (int m = 0; m < 8; ++m) s[m] = load_state4(p.initial_state, p.state_dtype, slot + m * kN);
    } else {
#pragma unroll
        for (int m = 0; m < 8; ++m) s[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const X *rp = static_cast<const X *>(p.r);
    const X *kp = static_cast<const X *>(p.k);
    const X *vp = static_cast<const X *>(p.v);
    const X *kkp = static_cast<const X *>(p.kk);
    const X *ap = static_cast<const X *>(p.a);
    const long long tok_stride = (long long)H * kN;

    TokenIn<X> cur, nxt;
    if (bos < eos)
        cur.load(rp, p.w, kp, vp, kkp, ap, bos * tok_stride + h * kN + row0,
                 bos * tok_stride + h * kN + col);
    for (int t = bos; t < eos; ++t) {
        if (t + 1 < eos)
            nxt.load(rp, p.w, kp, vp, kkp, ap, (t + 1) * tok_stride + h * kN + row0,
                     (t + 1) * tok_stride + h * kN + col);
        float rr[8], ww[8], kr[8], kkr[8], ar[8];
        cur.r.unpack(rr);
        cur.w.unpack(ww);
        cur.k.unpack(kr);
        cur.kk.unpack(kkr);
        cur.a.unpack(ar);

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
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float d = expf(ww[m]), c = kkr[m] * ar[m], kv = kr[m];
            s[m].x = fmaf(d, s[m].x, fmaf(-c, z0, kv * cur.v[0]));
            s[m].y = fmaf(d, s[m].y, fmaf(-c, z1, kv * cur.v[1]));
            s[m].z = fmaf(d, s[m].z, fmaf(-c, z2, kv * cur.v[2]));
            s[m].w = fmaf(d, s[m].w, fmaf(-c, z3, kv * cur.v[3]));
            o0 = fmaf(rr[m], s[m].x, o0);
            o1 = fmaf(rr[m], s[m].y, o1);
            o2 = fmaf(rr[m], s[m].z, o2);
            o3 = fmaf(rr[m], s[m].w, o3);
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            o0 += __shfl_xor_sync(0xffffffffu, o0, off);
            o1 += __shfl_xor_sync(0xffffffffu, o1, off);
            o2 += __shfl_xor_sync(0xffffffffu, o2, off);
            o3 += __shfl_xor_sync(0xffffffffu, o3, off);
        }
        if (rg == 0) {
            const long long at = t * tok_stride + h * kN + col;
            if (p.o_dtype == WKV7_BF16) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(o0, o1), hi = __floats2bfloat162_rn(o2, o3);
                uint2 u;
                u.x = *reinterpret_cast<const uint32_t *>(&lo);
                u.y = *reinterpret_cast<const uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.o) + at) = u;
            } else {
                *reinterpret_cast<float4 *>(static_cast<float *>(p.o) + at) = make_float4(o0, o1, o2, o3);
            }
        }
        cur = nxt;
    }

    if (p.final_state) {
#pragma unroll
        for (int m = 0; m < 8; ++m) store_state4(p.final_state, p.state_dtype, slot + m * kN, s[m]);
    }
}

}  // namespace

cudaError_t launch_prefill_scan(const PrefillArgs &args, cudaStream_t stream) {
    const long long pairs = (long long)args.num_seqs * args.H;
    if (pairs <= 0) return cudaSuccess;
    if (args.x_dtype == WKV7_BF16)
        wkv7_prefill_scan_kernel<__nv_bfloat16><<<(unsigned)pairs, kWarpsPerBlock * 32, 0, stream>>>(args);
    else
        wkv7_prefill_scan_kernel<float><<<(unsigned)pairs, kWarpsPerBlock * 32, 0, stream>>>(args);
    return cudaGetLastError();
}

}  // namespace wkv7
