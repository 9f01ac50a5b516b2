// Multi-token verify step for speculative decoding, and its rollback.
//
// One speculative step of the RWKV-Infer-Next page ("Inference. One speculative
// step"): the base model processes [t, d1 .. dK] in one forward, the sampler
// accepts the drafts up to the first mismatch, and the recurrent state is rolled
// back to the accepted prefix.  For the WKV part that is T = K + 1 consecutive
// decode steps per row from the current state, with every position's state kept
// so that the accepted one can be chosen afterwards:
//
//   S_{-1} = state ;  for t = 0 .. T-1:  S_t = step(S_{t-1}, x_t),  o_t = S_t^T r_t
//
// wkv7_verify_kernel: one head per CTA (four warps, the decode kernel's split:
// warp w owns value columns 16w .. 16w+15, lane L key rows 8 (L >> 2) .. +7 and
// four columns).  One thread bulk-copies the head's 16 KB state and the T
// tokens' six 256-byte vectors into shared memory; the state then stays in
// registers across the T tokens, and each S_t leaves from registers (16-byte
// stores, 64 contiguous bytes per key row and lane quad).
//
// wkv7_verify_commit_kernel: per head, copies S_{a-1} for the row's accepted
// length a (1 .. T) into the state; a = 0 leaves the state as it was.
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

using namespace ptx;

constexpr int kThreads = 128;
constexpr uint32_t kMaxPolls = 1u << 24;
constexpr int kMaxT = 8;

__device__ __forceinline__ float comp(const float4 &x, int c) {
    return c == 0 ? x.x : c == 1 ? x.y : c == 2 ? x.z : x.w;
}

// inputs [B, T, H, 64]; o [B, T, H, 64]; states [T, B, H, 64, 64]
__global__ void __launch_bounds__(kThreads)
wkv7_verify_kernel(int B, int T, int H, const float *__restrict__ r, const float *__restrict__ w,
                   const float *__restrict__ k, const float *__restrict__ v, const float *__restrict__ kk,
                   const float *__restrict__ a, const float *__restrict__ state, float *__restrict__ o,
                   float *__restrict__ states, unsigned *status) {
    extern __shared__ __align__(128) unsigned char smem[];
    float *S = reinterpret_cast<float *>(smem);                 // [64][64]
    float *vec = S + kN * kN;                                    // [T][6][64]
    unsigned long long *bar = reinterpret_cast<unsigned long long *>(vec + T * 6 * kN);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long head = blockIdx.x;  // b * H + h
    const long long b = head / H, h = head % H;

    // L2 prefetch of the head's state while the preceding grid finishes (L2 is coherent with
    // that grid's writes); nothing is loaded before it is done
    if (tid == 0) bulk_prefetch_l2(state + head * (kN * kN), kN * kN * 4);
    grid_dep_wait();
    if (tid == 0) {
        mbar_init(smem_addr(bar), 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(smem_addr(bar), kN * kN * 4 + static_cast<uint32_t>(T) * 6 * kN * 4);
        bulk_load(smem_addr(S), state + head * (kN * kN), kN * kN * 4, smem_addr(bar));
        const float *src[6] = {r, w, k, v, kk, a};
        for (int t = 0; t < T; ++t) {
            const long long row = ((b * T + t) * H + h) * kN;
#pragma unroll
            for (int i = 0; i < 6; ++i)
                bulk_load(smem_addr(vec + (t * 6 + i) * kN), src[i] + row, kN * 4, smem_addr(bar));
        }
    }
    __syncthreads();
    grid_dep_launch();
    const bool got = mbar_wait_bounded(smem_addr(bar), 0, kMaxPolls);
    if (__syncthreads_or(got ? 0 : 1)) {
        if (tid == 0) {
            report(status, kDevTimeout);
            mbar_wait_bounded(smem_addr(bar), 0, kMaxPolls);  // let the copies land before leaving
        }
        return;
    }

    const int rg = lane >> 2, row0 = rg * 8;
    const int col = warp * 16 + (lane & 3) * 4;
    float4 x[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) x[m] = *reinterpret_cast<const float4 *>(&S[(row0 + m) * kN + col]);

    for (int t = 0; t < T; ++t) {
        const float *V = vec + t * 6 * kN;
        const float4 r0 = *reinterpret_cast<const float4 *>(V + 0 * kN + row0);
        const float4 r1 = *reinterpret_cast<const float4 *>(V + 0 * kN + row0 + 4);
        const float4 w0 = *reinterpret_cast<const float4 *>(V + 1 * kN + row0);
        const float4 w1 = *reinterpret_cast<const float4 *>(V + 1 * kN + row0 + 4);
        const float4 k0 = *reinterpret_cast<const float4 *>(V + 2 * kN + row0);
        const float4 k1 = *reinterpret_cast<const float4 *>(V + 2 * kN + row0 + 4);
        const float4 vv = *reinterpret_cast<const float4 *>(V + 3 * kN + col);
        const float4 kk0 = *reinterpret_cast<const float4 *>(V + 4 * kN + row0);
        const float4 kk1 = *reinterpret_cast<const float4 *>(V + 4 * kN + row0 + 4);
        const float4 a0 = *reinterpret_cast<const float4 *>(V + 5 * kN + row0);
        const float4 a1 = *reinterpret_cast<const float4 *>(V + 5 * kN + row0 + 4);
        float kkr[8], kr[8], rr[8], dr[8], cr[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            kkr[m] = comp(kk0, m); kkr[m + 4] = comp(kk1, m);
            kr[m] = comp(k0, m);   kr[m + 4] = comp(k1, m);
            rr[m] = comp(r0, m);   rr[m + 4] = comp(r1, m);
            dr[m] = expf(comp(w0, m)); dr[m + 4] = expf(comp(w1, m));
            cr[m] = comp(kk0, m) * comp(a0, m); cr[m + 4] = comp(kk1, m) * comp(a1, m);
        }
        float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            z0 = fmaf(kkr[m], x[m].x, z0);
            z1 = fmaf(kkr[m], x[m].y, z1);
            z2 = fmaf(kkr[m], x[m].z, z2);
            z3 = fmaf(kkr[m], x[m].w, z3);
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            z0 += __shfl_xor_sync(0xffffffffu, z0, off);
            z1 += __shfl_xor_sync(0xffffffffu, z1, off);
            z2 += __shfl_xor_sync(0xffffffffu, z2, off);
            z3 += __shfl_xor_sync(0xffffffffu, z3, off);
        }
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
        float *St = states + (static_cast<long long>(t) * B * H + head) * (kN * kN) + row0 * kN + col;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float d = dr[m], c = cr[m], kv = kr[m];
            x[m].x = fmaf(d, x[m].x, fmaf(-c, z0, kv * vv.x));
            x[m].y = fmaf(d, x[m].y, fmaf(-c, z1, kv * vv.y));
            x[m].z = fmaf(d, x[m].z, fmaf(-c, z2, kv * vv.z));
            x[m].w = fmaf(d, x[m].w, fmaf(-c, z3, kv * vv.w));
            o0 = fmaf(rr[m], x[m].x, o0);
            o1 = fmaf(rr[m], x[m].y, o1);
            o2 = fmaf(rr[m], x[m].z, o2);
            o3 = fmaf(rr[m], x[m].w, o3);
            *reinterpret_cast<float4 *>(St + m * kN) = x[m];
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            o0 += __shfl_xor_sync(0xffffffffu, o0, off);
            o1 += __shfl_xor_sync(0xffffffffu, o1, off);
            o2 += __shfl_xor_sync(0xffffffffu, o2, off);
            o3 += __shfl_xor_sync(0xffffffffu, o3, off);
        }
        if (rg == 0)
            *reinterpret_cast<float4 *>(o + ((b * T + t) * H + h) * kN + col) = make_float4(o0, o1, o2, o3);
    }
}

// Grid: one CTA of 256 threads per head; copies states[a-1][head] to state[head].
__global__ void __launch_bounds__(256)
wkv7_verify_commit_kernel(int B, int T, int H, const float *__restrict__ states,
                          const int32_t *__restrict__ accept_len, float *__restrict__ state, unsigned *status) {
    grid_dep_wait();
    const long long head = blockIdx.x;
    const int b = static_cast<int>(head / H);
    const int acc = accept_len[b];
    if (acc < 0 || acc > T) {
        if (threadIdx.x == 0 && head % H == 0) report(status, kDevBounds);
        return;
    }
    if (acc == 0) return;
    const float4 *src = reinterpret_cast<const float4 *>(states + (static_cast<long long>(acc - 1) * B * H + head) * (kN * kN));
    float4 *dst = reinterpret_cast<float4 *>(state + head * (kN * kN));
    for (int e = threadIdx.x; e < kN * kN / 4; e += 256) dst[e] = src[e];
}

void set_pdl(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, cudaStream_t stream) {
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
}

}  // namespace

int verify_max_tokens() { return kMaxT; }

cudaError_t launch_verify(int B, int T, int H, const float *r, const float *w, const float *k, const float *v,
                          const float *kk, const float *a, const float *state, float *o, float *states,
                          unsigned *status, cudaStream_t stream) {
    const long long heads = static_cast<long long>(B) * H;
    if (heads <= 0 || T <= 0) return cudaSuccess;
    const size_t smem = (kN * kN + static_cast<size_t>(T) * 6 * kN) * sizeof(float) + 16;
    static int attr_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_dev != dev) {
        e = cudaFuncSetAttribute(wkv7_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>((kN * kN + kMaxT * 6 * kN) * sizeof(float) + 16));
        if (e != cudaSuccess) return e;
        attr_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl(cfg, attr, stream);
    cfg.gridDim = dim3(static_cast<unsigned>(heads));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, wkv7_verify_kernel, B, T, H, r, w, k, v, kk, a, state, o, states, status);
}

cudaError_t launch_verify_commit(int B, int T, int H, const float *states, const int32_t *accept_len, float *state,
                                 unsigned *status, cudaStream_t stream) {
    const long long heads = static_cast<long long>(B) * H;
    if (heads <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl(cfg, attr, stream);
    cfg.gridDim = dim3(static_cast<unsigned>(heads));
    cfg.blockDim = dim3(256);
    return cudaLaunchKernelEx(&cfg, wkv7_verify_commit_kernel, B, T, H, states, accept_len, state, status);
}

}  // namespace wkv7
