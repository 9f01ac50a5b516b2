// Decode step of the WKV-7 recurrence: one token for B*H heads, the fp32
// state read and written in place.
//
// Per head (Core AI model zoo note "Recurrent / linear-attention LLMs on
// Core AI", section 1), with S = [K, V]:
//     z = kk^T S ;  S' = diag(exp w) S - (kk .* a) z^T + k v^T ;  o = S'^T r
//
// The step moves 32 KB of state per head (read + write) against 1.8 KB of
// vectors: it is bound by HBM bandwidth, so the kernel is built around
// keeping enough bytes in flight on every SM regardless of register
// pressure.  It is persistent: CTA c owns heads c, c + G, c + 2G, ... (G =
// grid size, a multiple of the SM count), and streams them through a
// four-stage shared-memory ring.  One thread issues 1-D bulk async copies
// (the head's 16 KB state plus its six 256-byte input vectors) into a stage
// and the stage's mbarrier completes when the bytes land; the four warps
// compute; the new state goes back to global memory with one bulk async store
// from the same stage.  While one head is computed, the next three are in
// flight.
//
// Compute split (unchanged from the register form): the 64 value columns of a
// head evolve independently given the per-row vectors, so warp w owns columns
// 16w .. 16w+15; lane L holds key rows 8*(L>>2) .. +7 and columns 4*(L&3) ..
// +3 of that slice; the two reductions over key rows (kk^T S and S'^T r) are
// a per-lane sum over eight rows and three xor-shuffles.
//
// A register-resident form of the same computation (below) is used instead
// from 8192 heads per launch (many full waves: ~94% of measured bandwidth
// there) and when the launch fits in one wave of it (at most SMs x 6 heads:
// 912 on a GB300; 1.79 vs 2.11 us at 40 heads, 5.95 vs 6.89 us at 640).
// In between (e.g. 1280 heads: 9.25 vs 10.03 us) the ring is faster.
//
// Launch order: programmatic dependent launch.  The kernel waits for the
// preceding grid (griddepcontrol.wait) before it loads anything from global
// memory, so back-to-back calls on the same state stay ordered, while the
// launch and block scheduling of the next call overlap the tail of this one.
// Before the wait a block only issues L2 prefetches of the heads it will load
// first: they start the HBM reads during the preceding grid's tail, and since
// L2 is the point of coherence the loads after the wait still see every write
// of that grid.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

using namespace ptx;

constexpr int kThreads = 128;
constexpr int kStages = 4;
constexpr uint32_t kVecBytes = kN * 4;         // 256 B
constexpr uint32_t kMaxPolls = 1u << 24;

// One ring stage: a head's state and its vectors r, w, k, v, kk, a; with the fused
// time-mix tail also its gate g and the head's r_k, ln_w, ln_b.
template <bool kTail, typename ST = float>
struct Stage {
    static constexpr int kVecs = kTail ? 10 : 6;
    ST S[kN * kN];
    float vec[kVecs][kN];
};
static_assert(sizeof(Stage<false>) % 128 == 0 && sizeof(Stage<true>) % 128 == 0 &&
                  sizeof(Stage<false, __half>) % 128 == 0, "stage size");
template <bool kTail, typename ST = float>
constexpr size_t kSmemBytesT = kStages * sizeof(Stage<kTail, ST>) + kStages * sizeof(unsigned long long);
constexpr size_t kSmemBytes = kSmemBytesT<false>;
constexpr size_t kSmemBytes16 = kSmemBytesT<false, __half>;

// Four state elements (columns col .. col+3 of one row) of a ring stage, widened to
// fp32; and the store back, rounded to nearest even for the 16-bit types.
__device__ __forceinline__ float4 ld_state4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld_state4(const __half *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float4 ld_state4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ void st_state4(float *p, const float4 &x) { *reinterpret_cast<float4 *>(p) = x; }
__device__ __forceinline__ void st_state4(__half *p, const float4 &x) {
    const __half2 lo = __floats2half2_rn(x.x, x.y), hi = __floats2half2_rn(x.z, x.w);
    *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}
__device__ __forceinline__ void st_state4(__nv_bfloat16 *p, const float4 &x) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
    *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}

__device__ __forceinline__ float comp(const float4 &x, int c) {
    return c == 0 ? x.x : c == 1 ? x.y : c == 2 ? x.z : x.w;
}

// o[col .. col+3] of one head: fp32, or rounded to bf16 (to nearest even).
__device__ __forceinline__ void store_o4(float *__restrict__ o, long long idx, float o0, float o1, float o2,
                                         float o3) {
    *reinterpret_cast<float4 *>(o + idx) = make_float4(o0, o1, o2, o3);
}
__device__ __forceinline__ void store_o4(__nv_bfloat16 *__restrict__ o, long long idx, float o0, float o1,
                                         float o2, float o3) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(o0, o1), hi = __floats2bfloat162_rn(o2, o3);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&lo);
    u.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(o + idx) = u;
}

// The time-mix tail of one head in the decode layout (four warps; lane L of warp w holds
// key rows row0 .. row0+7 and value columns col .. col+3, and o0..o3 = o[col .. col+3],
// the same in every row group):
//   y = (GroupNorm_head(o) * ln_w + ln_b + (sum_i r_i k_i rk_i) v) * g
// In two halves around a block barrier.  tail_stats: the bonus (rk0, rk1 = r_k at rows
// row0 .. row0+7) by shuffles over the row groups, and this warp's mean and centred sum
// of squares over its 16 columns into red[warp], red[4 + warp].  tail_apply, after the
// barrier: the four merged (mean of means, plus 16 (m_w - m)^2 per warp), then y at
// columns col .. col+3 from ln_w (w4), ln_b (b4) and the gate (g4).
__device__ __forceinline__ float tail_stats(const float4 &rk0, const float4 &rk1, int warp, int lane,
                                            const float (&rr)[8], const float (&kr)[8], float o0, float o1,
                                            float o2, float o3, float *red) {
    float bonus = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        bonus = fmaf(rr[m] * kr[m], comp(rk0, m), bonus);
        bonus = fmaf(rr[m + 4] * kr[m + 4], comp(rk1, m), bonus);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) bonus += __shfl_xor_sync(0xffffffffu, bonus, off);
    float s1 = (o0 + o1) + (o2 + o3);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    const float mw = s1 * (1.f / 16);
    const float e0 = o0 - mw, e1 = o1 - mw, e2 = o2 - mw, e3 = o3 - mw;
    float q = fmaf(e0, e0, fmaf(e1, e1, fmaf(e2, e2, e3 * e3)));
    q += __shfl_xor_sync(0xffffffffu, q, 1);
    q += __shfl_xor_sync(0xffffffffu, q, 2);
    if (lane == 0) {
        red[warp] = mw;
        red[4 + warp] = q;
    }
    return bonus;
}

__device__ __forceinline__ float4 tail_apply(const float *red, float eps, float bonus, const float4 &w4,
                                             const float4 &b4, const float4 &g4, const float4 &vv, float o0,
                                             float o1, float o2, float o3) {
    const float m0 = red[0], m1 = red[1], m2 = red[2], m3 = red[3];
    const float mean = ((m0 + m1) + (m2 + m3)) * 0.25f;
    const float a0 = m0 - mean, a1 = m1 - mean, a2 = m2 - mean, a3 = m3 - mean;
    const float M2 = ((red[4] + red[5]) + (red[6] + red[7])) + 16.f * fmaf(a0, a0, fmaf(a1, a1, fmaf(a2, a2, a3 * a3)));
    const float rstd = rsqrtf(M2 * (1.f / kN) + eps);
    const float d0 = o0 - mean, d1 = o1 - mean, d2 = o2 - mean, d3 = o3 - mean;
    return make_float4((fmaf(d0 * rstd, w4.x, b4.x) + bonus * vv.x) * g4.x,
                       (fmaf(d1 * rstd, w4.y, b4.y) + bonus * vv.y) * g4.y,
                       (fmaf(d2 * rstd, w4.z, b4.z) + bonus * vv.z) * g4.z,
                       (fmaf(d3 * rstd, w4.w, b4.w) + bonus * vv.w) * g4.w);
}

template <bool kTail, typename OutT, typename ST = float>
__global__ void __launch_bounds__(kThreads)
wkv7_step_kernel(long long n_heads, const float *__restrict__ r, const float *__restrict__ w,
                 const float *__restrict__ k, const float *__restrict__ v,
                 const float *__restrict__ kk, const float *__restrict__ a,
                 ST *__restrict__ state, OutT *__restrict__ o, TailArgs tail, unsigned *status) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[2][8];  // the tail's statistics, double-buffered across heads
    using StageX = Stage<kTail, ST>;
    constexpr uint32_t kStBytes = kN * kN * sizeof(ST);
    StageX *st = reinterpret_cast<StageX *>(smem);
    unsigned long long *full = reinterpret_cast<unsigned long long *>(smem + kStages * sizeof(StageX));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const long long first = blockIdx.x, stride = gridDim.x;
    const long long count = n_heads > first ? (n_heads - 1 - first) / stride + 1 : 0;
    const float *const vsrc[6] = {r, w, k, v, kk, a};

    // While the preceding grid finishes, its tail overlaps with L2 prefetches of the heads
    // this block loads first (prefetches read nothing into the block and L2 is coherent
    // with that grid's writes).  Nothing is loaded before the preceding grid is done.
    if (tid == 0) {
        for (long long idx = 0; idx < count && idx < kStages; ++idx) {
            const long long head = first + idx * stride;
            bulk_prefetch_l2(state + head * (kN * kN), kStBytes);
#pragma unroll
            for (int i = 0; i < 6; ++i) bulk_prefetch_l2(vsrc[i] + head * kN, kVecBytes);
        }
    }
    grid_dep_wait();
    auto issue = [&](long long idx) {
        const long long head = first + idx * stride;
        const int s = static_cast<int>(idx % kStages);
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, kStBytes + StageX::kVecs * kVecBytes);
        bulk_load(smem_addr(st[s].S), state + head * (kN * kN), kStBytes, bar);
#pragma unroll
        for (int i = 0; i < 6; ++i) bulk_load(smem_addr(st[s].vec[i]), vsrc[i] + head * kN, kVecBytes, bar);
        if constexpr (kTail) {
            const long long hp = head % tail.H;
            bulk_load(smem_addr(st[s].vec[6]), static_cast<const float *>(tail.g) + head * kN, kVecBytes, bar);
            bulk_load(smem_addr(st[s].vec[7]), tail.rk + hp * kN, kVecBytes, bar);
            bulk_load(smem_addr(st[s].vec[8]), tail.ln_w + hp * kN, kVecBytes, bar);
            bulk_load(smem_addr(st[s].vec[9]), tail.ln_b + hp * kN, kVecBytes, bar);
        }
    };
    // thread 0 sets up the barriers and starts the first loads before the block syncs
    long long issued = 0;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&full[s]), 1);
        fence_mbar_init();
        for (; issued < count && issued < kStages; ++issued) issue(issued);
    }
    __syncthreads();
    grid_dep_launch();

    const int rg = lane >> 2;
    const int row0 = rg * 8;
    const int col = warp * 16 + (lane & 3) * 4;
    long long failed_at = -1;
    for (long long idx = 0; idx < count; ++idx) {
        const int s = static_cast<int>(idx % kStages);
        const uint32_t parity = static_cast<uint32_t>((idx / kStages) & 1);
        const bool got = mbar_wait_bounded(smem_addr(&full[s]), parity, kMaxPolls);
        if (__syncthreads_or(got ? 0 : 1)) {
            failed_at = idx;
            break;
        }
        const long long head = first + idx * stride;
        StageX &S = st[s];

        float4 x[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) x[m] = ld_state4(&S.S[(row0 + m) * kN + col]);
        const float4 r0 = *reinterpret_cast<const float4 *>(&S.vec[0][row0]);
        const float4 r1 = *reinterpret_cast<const float4 *>(&S.vec[0][row0 + 4]);
        const float4 w0 = *reinterpret_cast<const float4 *>(&S.vec[1][row0]);
        const float4 w1 = *reinterpret_cast<const float4 *>(&S.vec[1][row0 + 4]);
        const float4 k0 = *reinterpret_cast<const float4 *>(&S.vec[2][row0]);
        const float4 k1 = *reinterpret_cast<const float4 *>(&S.vec[2][row0 + 4]);
        const float4 vv = *reinterpret_cast<const float4 *>(&S.vec[3][col]);
        const float4 kk0 = *reinterpret_cast<const float4 *>(&S.vec[4][row0]);
        const float4 kk1 = *reinterpret_cast<const float4 *>(&S.vec[4][row0 + 4]);
        const float4 a0 = *reinterpret_cast<const float4 *>(&S.vec[5][row0]);
        const float4 a1 = *reinterpret_cast<const float4 *>(&S.vec[5][row0 + 4]);

        float kkr[8], kr[8], rr[8], dr[8], cr[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            kkr[m] = comp(kk0, m); kkr[m + 4] = comp(kk1, m);
            kr[m] = comp(k0, m);   kr[m + 4] = comp(k1, m);
            rr[m] = comp(r0, m);   rr[m + 4] = comp(r1, m);
            dr[m] = expf(comp(w0, m)); dr[m + 4] = expf(comp(w1, m));
            cr[m] = comp(kk0, m) * comp(a0, m); cr[m + 4] = comp(kk1, m) * comp(a1, m);
        }
        // z = kk^T S over the old state
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
        // S' = diag(exp w) S - (kk .* a) z^T + k v^T, then o = S'^T r
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
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
            st_state4(&S.S[(row0 + m) * kN + col], x[m]);
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            o0 += __shfl_xor_sync(0xffffffffu, o0, off);
            o1 += __shfl_xor_sync(0xffffffffu, o1, off);
            o2 += __shfl_xor_sync(0xffffffffu, o2, off);
            o3 += __shfl_xor_sync(0xffffffffu, o3, off);
        }
        float bonus = 0.f;
        if constexpr (kTail) {
            bonus = tail_stats(*reinterpret_cast<const float4 *>(&S.vec[7][row0]),
                               *reinterpret_cast<const float4 *>(&S.vec[7][row0 + 4]), warp, lane, rr, kr, o0, o1,
                               o2, o3, red[idx & 1]);
            if (o && rg == 0) store_o4(o, head * kN + col, o0, o1, o2, o3);
        } else if (rg == 0) {
            // the fp32 store written out here: through the helper this kernel ran 2.5% slower
            if constexpr (sizeof(OutT) == 4)
                *reinterpret_cast<float4 *>(o + head * kN + col) = make_float4(o0, o1, o2, o3);
            else
                store_o4(o, head * kN + col, o0, o1, o2, o3);
        }

        fence_proxy_async_smem();  // the new state in this stage -> visible to the bulk store
        __syncthreads();           // (and the tail's statistics of every warp)
        if constexpr (kTail) {
            const float4 y = tail_apply(red[idx & 1], tail.eps, bonus, *reinterpret_cast<const float4 *>(&S.vec[8][col]),
                                        *reinterpret_cast<const float4 *>(&S.vec[9][col]),
                                        *reinterpret_cast<const float4 *>(&S.vec[6][col]), vv, o0, o1, o2, o3);
            if (rg == 0) *reinterpret_cast<float4 *>(tail.y + head * kN + col) = y;
        }
        if (tid == 0) {
            bulk_store(state + head * (kN * kN), smem_addr(S.S), kStBytes);
            bulk_commit();
            // refill the previous stage once its store has read it
            if (idx >= 1 && issued < count) {
                bulk_wait_read<1>();
                issue(issued);
                ++issued;
            }
        }
    }
    if (tid == 0) {
        if (failed_at >= 0) {
            report(status, kDevTimeout);
            // let every load still outstanding land before the CTA's shared memory goes away
            for (long long idx = failed_at; idx < issued; ++idx)
                mbar_wait_bounded(smem_addr(&full[idx % kStages]), static_cast<uint32_t>((idx / kStages) & 1),
                                  kMaxPolls);
        }
        // the last state stores have read shared memory; their writes are complete when the
        // grid is (which is what the next dependent launch waits for)
        bulk_wait_read<0>();
    }
}

// Register-resident variant for large batches: one warp per 16-column slice,
// the eight float4 words of state per lane loaded straight into registers.
// With thousands of heads per launch the grid runs many full waves, so the
// occupancy limit of this form (24 warps/SM at 80 registers) costs nothing,
// and it avoids the per-head shared-memory round trip of the ring above.
constexpr int kRegWarps = 4;

template <bool kTail, typename OutT>
__global__ void __launch_bounds__(kRegWarps * 32)
wkv7_step_regs_kernel(long long n_units, const float *__restrict__ r, const float *__restrict__ w,
                      const float *__restrict__ k, const float *__restrict__ v,
                      const float *__restrict__ kk, const float *__restrict__ a,
                      float *__restrict__ state, OutT *__restrict__ o, TailArgs tail) {
    __shared__ float red[8];  // a block is the four slices of one head
    const int lane = threadIdx.x & 31;
    const long long unit = static_cast<long long>(blockIdx.x) * kRegWarps + (threadIdx.x >> 5);
    // L2 prefetch of this block's head while the preceding grid finishes (as in the ring form)
    if (threadIdx.x == 0 && unit < n_units) {
        const long long hd = unit >> 2;
        bulk_prefetch_l2(state + hd * (kN * kN), kN * kN * 4);
        const float *const vsrc[6] = {r, w, k, v, kk, a};
#pragma unroll
        for (int i = 0; i < 6; ++i) bulk_prefetch_l2(vsrc[i] + hd * kN, kVecBytes);
    }
    grid_dep_wait();
    if (unit >= n_units) return;
    const long long head = unit >> 2;
    const int slice = static_cast<int>(unit & 3);
    const int rg = lane >> 2, row0 = rg * 8;
    const int col = slice * 16 + (lane & 3) * 4;
    float *S = state + head * (kN * kN) + static_cast<long long>(row0) * kN + col;
    float4 x[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) x[m] = *reinterpret_cast<const float4 *>(S + m * kN);
    // the next grid may be scheduled once every block has its state (triggering at the
    // start instead: B = 8 on the 2.9B geometry 3.10 -> 3.93 us)
    grid_dep_launch();
    const long long vb = head * kN + row0;
    const float4 r0 = __ldg(reinterpret_cast<const float4 *>(r + vb)), r1 = __ldg(reinterpret_cast<const float4 *>(r + vb + 4));
    const float4 w0 = __ldg(reinterpret_cast<const float4 *>(w + vb)), w1 = __ldg(reinterpret_cast<const float4 *>(w + vb + 4));
    const float4 k0 = __ldg(reinterpret_cast<const float4 *>(k + vb)), k1 = __ldg(reinterpret_cast<const float4 *>(k + vb + 4));
    const float4 kk0 = __ldg(reinterpret_cast<const float4 *>(kk + vb)), kk1 = __ldg(reinterpret_cast<const float4 *>(kk + vb + 4));
    const float4 a0 = __ldg(reinterpret_cast<const float4 *>(a + vb)), a1 = __ldg(reinterpret_cast<const float4 *>(a + vb + 4));
    const float4 vv = __ldg(reinterpret_cast<const float4 *>(v + head * kN + col));
    // the tail's vectors, fetched now so that their latency hides behind the state math
    float4 pre[5];
    if constexpr (kTail) {
        const long long hp = head % tail.H;
        pre[0] = __ldg(reinterpret_cast<const float4 *>(tail.rk + hp * kN + row0));
        pre[1] = __ldg(reinterpret_cast<const float4 *>(tail.rk + hp * kN + row0 + 4));
        pre[2] = __ldg(reinterpret_cast<const float4 *>(tail.ln_w + hp * kN + col));
        pre[3] = __ldg(reinterpret_cast<const float4 *>(tail.ln_b + hp * kN + col));
        pre[4] = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(tail.g) + head * kN + col));
    }
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
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) *reinterpret_cast<float4 *>(S + m * kN) = x[m];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        o0 += __shfl_xor_sync(0xffffffffu, o0, off);
        o1 += __shfl_xor_sync(0xffffffffu, o1, off);
        o2 += __shfl_xor_sync(0xffffffffu, o2, off);
        o3 += __shfl_xor_sync(0xffffffffu, o3, off);
    }
    if constexpr (kTail) {
        const float bonus = tail_stats(pre[0], pre[1], slice, lane, rr, kr, o0, o1, o2, o3, red);
        __syncthreads();
        const float4 y = tail_apply(red, tail.eps, bonus, pre[2], pre[3], pre[4], vv, o0, o1, o2, o3);
        if (rg == 0) *reinterpret_cast<float4 *>(tail.y + head * kN + col) = y;
        if (o && rg == 0) store_o4(o, head * kN + col, o0, o1, o2, o3);
    } else {
        if (rg == 0) store_o4(o, head * kN + col, o0, o1, o2, o3);
    }
}

// ---------------------------------------------------------------- 16-bit state
//
// The same step with the state stored in fp16 or bf16 (wkv7_step_kernel with
// ST = __half or __nv_bfloat16): the bulk copies move 8 KB per head instead of
// 16 KB, each element is widened to fp32 when it is read from the ring stage,
// the whole update and read-out run in fp32, and the new state is rounded to
// nearest even when it is written back into the stage, from where the bulk
// store takes it.  The Core AI model zoo note (section 5, "Parity gate +
// tokenizer") runs an fp16 export with fp16 state arrays; the state traffic,
// 95% of a decode step's bytes, halves.  The ring is used for every head count:
// staged in shared memory, a stage's bytes in flight do not depend on registers,
// which hold only half as many state bytes in 16 bits.

// Head count from which the register form is used (several full waves).
constexpr long long kRegsFromHeads = 8192;

struct LaunchShape {
    int grid_cap = 0;       // CTAs per wave (SMs x resident CTAs per SM)
    int grid_cap_tail = 0;  // the same for the form with the fused tail
    long long regs_wave = 0;  // heads the register-resident form runs in one wave
};

LaunchShape shape_for_device() {
    static int cached_dev = -1;
    static LaunchShape cached;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LaunchShape{};
    if (dev == cached_dev) return cached;
    LaunchShape s;
    int sms = 0, per_sm = 0;
    int per_sm_tail = 0;
    if (cudaFuncSetAttribute(wkv7_step_kernel<false, float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(wkv7_step_kernel<true, float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytesT<true>)) != cudaSuccess ||
        cudaFuncSetAttribute(wkv7_step_kernel<false, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, wkv7_step_kernel<false, float>, kThreads, kSmemBytes) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_tail, wkv7_step_kernel<true, float>, kThreads,
                                                      kSmemBytesT<true>) != cudaSuccess)
        return LaunchShape{};
    int per_sm_regs = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_regs, wkv7_step_regs_kernel<false, float>, kRegWarps * 32, 0) !=
        cudaSuccess)
        return LaunchShape{};
    s.regs_wave = static_cast<long long>(sms) * (per_sm_regs > 0 ? per_sm_regs : 1);
    s.grid_cap_tail = sms * (per_sm_tail > 0 ? per_sm_tail : 1);
    s.grid_cap = sms * (per_sm > 0 ? per_sm : 1);
    cached = s;
    cached_dev = dev;
    return s;
}

}  // namespace

cudaError_t launch_step_state16(long long n_heads, const float *r, const float *w, const float *k, const float *v,
                                const float *kk, const float *a, void *state, wkv7_dtype state_dtype, void *o,
                                wkv7_dtype o_dtype, unsigned *status, cudaStream_t stream) {
    if (n_heads <= 0) return cudaSuccess;
    static int cached_dev = -1, cap = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != cached_dev) {
        int sms = 0, per_sm = 0;
        const void *fns[4] = {reinterpret_cast<const void *>(wkv7_step_kernel<false, float, __half>),
                              reinterpret_cast<const void *>(wkv7_step_kernel<false, __nv_bfloat16, __half>),
                              reinterpret_cast<const void *>(wkv7_step_kernel<false, float, __nv_bfloat16>),
                              reinterpret_cast<const void *>(wkv7_step_kernel<false, __nv_bfloat16, __nv_bfloat16>)};
        for (const void *f : fns) {
            e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes16));
            if (e != cudaSuccess) return e;
        }
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, wkv7_step_kernel<false, float, __half>, kThreads,
                                                          kSmemBytes16);
        if (e != cudaSuccess) return e;
        cap = sms * (per_sm > 0 ? per_sm : 1);
        cached_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(n_heads < cap ? n_heads : cap));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes16;
    const TailArgs t{};
    const bool ob = o_dtype == WKV7_BF16;
    if (state_dtype == WKV7_F16) {
        if (ob) return cudaLaunchKernelEx(&cfg, wkv7_step_kernel<false, __nv_bfloat16, __half>, n_heads, r, w, k, v, kk, a, static_cast<__half *>(state), static_cast<__nv_bfloat16 *>(o), t, status);
        return cudaLaunchKernelEx(&cfg, wkv7_step_kernel<false, float, __half>, n_heads, r, w, k, v, kk, a, static_cast<__half *>(state), static_cast<float *>(o), t, status);
    }
    if (ob) return cudaLaunchKernelEx(&cfg, wkv7_step_kernel<false, __nv_bfloat16, __nv_bfloat16>, n_heads, r, w, k, v, kk, a, static_cast<__nv_bfloat16 *>(state), static_cast<__nv_bfloat16 *>(o), t, status);
    return cudaLaunchKernelEx(&cfg, wkv7_step_kernel<false, float, __nv_bfloat16>, n_heads, r, w, k, v, kk, a, static_cast<__nv_bfloat16 *>(state), static_cast<float *>(o), t, status);
}

cudaError_t launch_step(long long n_heads, const float *r, const float *w, const float *k,
                        const float *v, const float *kk, const float *a, float *state,
                        void *o, wkv7_dtype o_dtype, const TailArgs *tail, unsigned *status,
                        cudaStream_t stream) {
    const bool bf16 = o_dtype == WKV7_BF16;
    const TailArgs t = tail ? *tail : TailArgs{};
    if (n_heads <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const LaunchShape shape = shape_for_device();
    if (shape.grid_cap <= 0) return cudaErrorInvalidDevice;
    // The register-resident form whenever the launch is one wave of it (a head per
    // 4-warp block: no ring to fill, every head's loads issued at once) or many waves.
    if (n_heads >= kRegsFromHeads || n_heads <= shape.regs_wave) {
        const long long units = n_heads * 4;
        cfg.gridDim = dim3(static_cast<unsigned>((units + kRegWarps - 1) / kRegWarps));
        cfg.blockDim = dim3(kRegWarps * 32);
        if (tail) return cudaLaunchKernelEx(&cfg, wkv7_step_regs_kernel<true, float>, units, r, w, k, v, kk, a, state, static_cast<float *>(o), t);
        if (bf16) return cudaLaunchKernelEx(&cfg, wkv7_step_regs_kernel<false, __nv_bfloat16>, units, r, w, k, v, kk, a, state, static_cast<__nv_bfloat16 *>(o), t);
        return cudaLaunchKernelEx(&cfg, wkv7_step_regs_kernel<false, float>, units, r, w, k, v, kk, a, state, static_cast<float *>(o), t);
    }
    const long long cap = tail ? shape.grid_cap_tail : shape.grid_cap;
    const long long grid = n_heads < cap ? n_heads : cap;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = tail ? kSmemBytesT<true> : kSmemBytes;
    if (tail) return cudaLaunchKernelEx(&cfg, wkv7_step_kernel<true, float>, n_heads, r, w, k, v, kk, a, state, static_cast<float *>(o), t, status);
    if (bf16) return cudaLaunchKernelEx(&cfg, wkv7_step_kernel<false, __nv_bfloat16>, n_heads, r, w, k, v, kk, a, state, static_cast<__nv_bfloat16 *>(o), t, status);
    return cudaLaunchKernelEx(&cfg, wkv7_step_kernel<false, float>, n_heads, r, w, k, v, kk, a, state, static_cast<float *>(o), t, status);
}

}  // namespace wkv7
