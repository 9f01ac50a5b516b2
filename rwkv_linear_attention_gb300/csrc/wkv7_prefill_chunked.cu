// Chunked prefill of the WKV-7 recurrence on tcgen05 tensor cores.
//
// The per-token update (Core AI model zoo note "Recurrent / linear-attention
// LLMs on Core AI", section 1), per head with S = [K, V]:
//     z_t = S_{t-1}^T kk_t ;  S_t = D_t S_{t-1} - c_t z_t^T + k_t v_t^T ;  o_t = S_t^T r_t
// with D_t = diag(exp w_t), c_t = kk_t * a_t, is regrouped over chunks of
// C = 64 tokens.  With g_t = sum_{u<=t} w_u (inclusive, per key channel,
// restarted at the chunk start) the chunk's 64 projections z_t solve a unit
// lower-triangular system, and the whole chunk becomes
//
//   L_c[t,s] = sum_i kk_t[i] c_s[i] e^{g_{t-1}[i]-g_s[i]}   (s <  t)
//   L_k[t,s] = sum_i kk_t[i] k_s[i] e^{g_{t-1}[i]-g_s[i]}   (s <  t)
//   M_c[t,s] = sum_i r_t[i]  c_s[i] e^{g_t[i]-g_s[i]}       (s <= t)
//   M_k[t,s] = sum_i r_t[i]  k_s[i] e^{g_t[i]-g_s[i]}       (s <= t)
//   T = (I + L_c)^{-1}                       (the UT transform)
//   Z = T (Qa S0 + L_k V),   Qa[t,i] = kk_t[i] e^{g_{t-1}[i]}
//   O = Ra S0 + M_k V - M_c Z,               Ra[t,i] = r_t[i] e^{g_t[i]}
//   S_C = diag(e^{g_C}) S0 + Kb^T V - Cb^T Z,   Kb[s,i] = k_s[i] e^{g_C[i]-g_s[i]}, Cb likewise
//
// Substituting Z and folding every state-independent product gives one
// matrix product per chunk on the state's critical path:
//
//   [ O                     ]   [ Ra - Mt Qa   | M_k - Mt L_k  ]   [ S0 ]
//   [ S_C - e^{g_C} * S0    ] = [ -Ct Qa       | Kb^T - Ct L_k ] . [ V  ]
//
// with Mt = M_c T and Ct = Cb^T T.  Per chunk this kernel runs four tf32
// MMAs, all M = 128 with fp32 accumulators in tensor memory:
//   G  = [R ; Q] [C ; K]^T      (the four Gram blocks at once; 128x128x64)
//   X  = [M_c ; Cb^T] T         ([Mt ; Ct]; 128x64x64)
//   Y  = X [Qa | L_k]           (128x128x64)
//   D  = A_chain [S0 ; V]       (128x64x128)
// Everything else (cumulative decay, the exponentials, masks, the blocked
// 64x64 unit-lower-triangular inverse, operand staging) is SIMT work on the
// same CTA.  One CTA owns one (sequence, head) pair and walks its chunks in
// order; the fp32 state lives in registers between chunks.  Inputs arrive by
// TMA (2-D tiles of 64 tokens x 64 channels of the packed [T, H, 64] arrays);
// the next chunk's tiles load while the current chunk's last phases run.
//
// Inputs r, k, v, kk, a are bf16 (w fp32); fp32-input prefill is served by
// the token-serial kernel instead.
//
// Precision: inputs are used exactly; every MMA operand is rounded to tf32
// (round to nearest) and accumulates in fp32.  The decay factors of the Gram
// operands are taken relative to the chunk's middle token, so for
// w >= -2.5 every factor lies within e^{+-80} (finite in fp32).
#include <cuda.h>
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"
#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk length
constexpr int kThreads = 256;   // warp w reads TMEM lanes 32*(w%4).., column half w/4
constexpr uint32_t kMaxPolls = 1u << 24;

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0, kColX = 128, kColY = 192, kColD = 320;

// LC / TS scratch: fp32 64 x 68 (row stride 272 B keeps float4 rows conflict-free)
constexpr int kLd = 68;

template <int XB>
struct Layout {
    static constexpr int kTile = 64 * 64 * XB;     // one raw x tile
    static constexpr int R = 0;
    static constexpr int K = R + kTile;
    static constexpr int KK = K + kTile;
    static constexpr int A = KK + kTile;
    static constexpr int W = A + kTile;            // fp32 w -> cumulative g -> E = e^{g - g_ref}
    static constexpr int AX = W + 16384;           // 32 KB: [M_c ; Cb^T] operand; earlier LC scratch, raw v tile at +16 KB
    static constexpr int BX = AX + 32768;          // 16 KB: T^T operand
    static constexpr int P = BX + 16384;           // 64 KB: [A_G | B_G] -> TS/X scratch + B_Y -> [A_Y | B_Y] -> A_chain
    static constexpr int BC = P + 65536;           // 32 KB: B_chain = [S0^T | V^T] (64 rows x K 128)
    static constexpr int MISC = BC + 32768;        // per-channel vectors, barriers
    static constexpr int M_EREF = MISC;            // 64 f32: e^{g_ref}
    static constexpr int M_GC = MISC + 256;        // 64 f32: e^{g_C}
    static constexpr int M_TOT = MISC + 512;       // 4 x 64 f32: cumsum partials
    static constexpr int M_BAR_TMA = MISC + 1536;
    static constexpr int M_BAR_MMA = MISC + 1544;
    static constexpr int M_SLOT = MISC + 1552;
    static constexpr int kBytes = MISC + 1600;
    static constexpr int kAlloc = kBytes + 1024;   // slack to align the base to 1024 B
    static constexpr uint32_t kTmaBytes = 5 * kTile + 16384;
};
static_assert(Layout<2>::kAlloc <= 232448, "layout exceeds shared memory");

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void st_tf32x4(unsigned char *p, float a, float b, float c, float d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(to_tf32(a), to_tf32(b), to_tf32(c), to_tf32(d));
}
// Reciprocal of a decay factor (fast approximate divide, ~2 ulp).  Its
// result only feeds tf32 operands, whose rounding (2^-11) dominates.
__device__ __forceinline__ float rcp(float x) { return __fdividef(1.f, x); }
__device__ __forceinline__ float4 ld_f4(const unsigned char *p) {
    return *reinterpret_cast<const float4 *>(p);
}

// Raw input access (row-major [64 tokens][64 channels] tile of x).
template <typename X>
struct Raw;
template <>
struct Raw<__nv_bfloat16> {
    static constexpr int kB = 2;
    __device__ static float4 ld4(const unsigned char *tile, int t, int i) {
        const uint2 u = *reinterpret_cast<const uint2 *>(tile + (t * 64 + i) * 2);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    __device__ static float ld1(const unsigned char *tile, int t, int i) {
        const unsigned short u = *reinterpret_cast<const unsigned short *>(tile + (t * 64 + i) * 2);
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    }
};

struct TensorMaps {
    CUtensorMap r, k, v, kk, a, w;
};

// All threads wait on an mbarrier phase; the outcome is made uniform so that
// either every thread continues or every thread leaves together.
__device__ __forceinline__ bool wait_uniform(uint32_t bar, uint32_t parity, unsigned *status) {
    const bool ok = mbar_wait_bounded(bar, parity, kMaxPolls);
    const int any_fail = __syncthreads_or(ok ? 0 : 1);
    if (any_fail && threadIdx.x == 0) report(status, kDevTimeout);
    return any_fail == 0;
}

__device__ __forceinline__ void sync_for_mma() {
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
}

template <typename X>
__global__ void __launch_bounds__(kThreads, 1)
wkv7_prefill_chunked_kernel(PrefillArgs p, const __grid_constant__ TensorMaps maps) {
    using L = Layout<Raw<X>::kB>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q = warp & 3, hf = warp >> 2;  // TMEM lane quarter, column half
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;

    const int H = p.H;
    const int rank = static_cast<int>(blockIdx.x) / H;
    const int h = static_cast<int>(blockIdx.x) % H;
    const int b = p.order ? p.order[rank] : rank;
    if (b < 0 || b >= p.num_seqs) {
        if (tid == 0) report(p.status, kDevBounds);
        return;
    }
    const int bos = p.cu_seqlens[b], eos = p.cu_seqlens[b + 1];
    if (bos < 0 || eos < bos || eos > p.T_total) {
        if (tid == 0) report(p.status, kDevBadSeqlens);
        return;
    }
    const int len = eos - bos;
    const int nchunks = (len + kC - 1) / kC;
    const long long tok_stride = static_cast<long long>(H) * 64;
    float *eref = reinterpret_cast<float *>(sm + L::M_EREF);
    float *gC = reinterpret_cast<float *>(sm + L::M_GC);
    const uint32_t bar_tma = sbase + L::M_BAR_TMA, bar_mma = sbase + L::M_BAR_MMA;

    // State rows held by warps with q in {2, 3}: row i, columns [32*hf, 32*hf+32).
    const bool state_thread = q >= 2;
    const int srow = 32 * (q - 2) + lane;
    float s[32];
    const long long sslot = (static_cast<long long>(b) * H + h) * 4096;
    if (state_thread) {
        if (p.initial_state) {
            const float4 *src = reinterpret_cast<const float4 *>(p.initial_state + sslot + srow * 64 + 32 * hf);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 x = src[j];
                s[4 * j] = x.x; s[4 * j + 1] = x.y; s[4 * j + 2] = x.z; s[4 * j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) s[j] = 0.f;
        }
    }
    if (nchunks == 0) {
        if (state_thread && p.final_state) {
            float4 *dst = reinterpret_cast<float4 *>(p.final_state + sslot + srow * 64 + 32 * hf);
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]);
        }
        return;
    }

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(sbase + L::M_SLOT, kTmemCols);
    // B_chain rows j, K 0..63 <- S0[i][j] (tf32)
    if (state_thread) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            *reinterpret_cast<uint32_t *>(sm + L::BC + sw128_off(32 * hf + j, srow, 64)) = to_tf32(s[j]);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + L::M_SLOT);

    auto issue_tma = [&](int chunk) {
        const int y = bos + chunk * kC;
        const int x = h * 64;
        mbar_arrive_expect_tx(bar_tma, L::kTmaBytes);
        tma_load_2d(sbase + L::R, &maps.r, x, y, bar_tma);
        tma_load_2d(sbase + L::K, &maps.k, x, y, bar_tma);
        tma_load_2d(sbase + L::KK, &maps.kk, x, y, bar_tma);
        tma_load_2d(sbase + L::A, &maps.a, x, y, bar_tma);
        tma_load_2d(sbase + L::W, &maps.w, x, y, bar_tma);
        tma_load_2d(sbase + L::AX + 16384, &maps.v, x, y, bar_tma);
    };
    if (tid == 0) issue_tma(0);

    uint32_t mma_parity = 0;
    bool alive = true;
    using RawX = Raw<X>;
    unsigned char *rr = sm + L::R, *rk = sm + L::K, *rkk = sm + L::KK, *ra = sm + L::A, *rv = sm + L::AX + 16384;
    float *Et = reinterpret_cast<float *>(sm + L::W);  // [64][64]

    for (int c = 0; c < nchunks && alive; ++c) {
        const int t0 = bos + c * kC;
        const int lc = min(kC, eos - t0);

        if (!wait_uniform(bar_tma, static_cast<uint32_t>(c & 1), p.status)) { alive = false; break; }

        // ---- phase 2a: masked cumulative log-decay g (in place in the w tile)
        {
            const int ch = tid & 63, qq = tid >> 6;
            float g[16];
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = 16 * qq + u;
                acc += (t < lc) ? Et[t * 64 + ch] : 0.f;
                g[u] = acc;
            }
            float *tot = reinterpret_cast<float *>(sm + L::M_TOT);
            tot[qq * 64 + ch] = acc;
            __syncthreads();
            float pre = 0.f;
            for (int u = 0; u < qq; ++u) pre += tot[u * 64 + ch];
#pragma unroll
            for (int u = 0; u < 16; ++u) Et[(16 * qq + u) * 64 + ch] = pre + g[u];
            __syncthreads();
            // ---- phase 2b: E = e^{g - g_ref}, g_ref = g[31]; eref = e^{g_ref}
            const float gr = Et[31 * 64 + ch];
            __syncthreads();
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = 16 * qq + u;
                Et[t * 64 + ch] = __expf(Et[t * 64 + ch] - gr);
            }
            if (qq == 0) eref[ch] = __expf(gr);
            __syncthreads();
        }

        // ---- phase 2c: Gram operands A_G = [R ; Q] (rows t), B_G = [C ; K] (rows s), V^T into B_chain
        {
            unsigned char *AG = sm + L::P, *BG = sm + L::P + 32768;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int task = tid + kThreads * m;
                const int t = task >> 4, i = (task & 15) * 4;
                const float valid = t < lc ? 1.f : 0.f;
                const float4 e = ld_f4(reinterpret_cast<unsigned char *>(Et + t * 64 + i));
                float4 ep;  // e^{g_{t-1} - g_ref}
                if (t > 0) {
                    ep = ld_f4(reinterpret_cast<unsigned char *>(Et + (t - 1) * 64 + i));
                } else {
                    ep = make_float4(rcp(eref[i]), rcp(eref[i + 1]), rcp(eref[i + 2]), rcp(eref[i + 3]));
                }
                const float4 xr = RawX::ld4(rr, t, i), xk = RawX::ld4(rk, t, i);
                const float4 xkk = RawX::ld4(rkk, t, i), xa = RawX::ld4(ra, t, i);
                st_tf32x4(AG + sw128_off(t, i, 128), valid * xr.x * e.x, valid * xr.y * e.y,
                          valid * xr.z * e.z, valid * xr.w * e.w);
                st_tf32x4(AG + sw128_off(64 + t, i, 128), valid * xkk.x * ep.x, valid * xkk.y * ep.y,
                          valid * xkk.z * ep.z, valid * xkk.w * ep.w);
                const float4 ei = make_float4(valid * rcp(e.x), valid * rcp(e.y), valid * rcp(e.z), valid * rcp(e.w));
                st_tf32x4(BG + sw128_off(t, i, 128), xkk.x * xa.x * ei.x, xkk.y * xa.y * ei.y,
                          xkk.z * xa.z * ei.z, xkk.w * xa.w * ei.w);
                st_tf32x4(BG + sw128_off(64 + t, i, 128), xk.x * ei.x, xk.y * ei.y, xk.z * ei.z, xk.w * ei.w);
            }
            // V^T: B_chain[j][64 + s] = v[s][j]
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int j = tid & 63, sc = (tid >> 6) + 4 * m, s0 = 4 * sc;
                float vv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) vv[e] = (s0 + e < lc) ? RawX::ld1(rv, s0 + e, j) : 0.f;
                st_tf32x4(sm + L::BC + sw128_off(j, 64 + s0, 64), vv[0], vv[1], vv[2], vv[3]);
            }
        }
        sync_for_mma();

        // ---- MMA G: [R ; Q] x [C ; K]^T -> TMEM G (128 x 128)
        if (tid == 0) {
#pragma unroll
            for (int kq = 0; kq < 8; ++kq) {
                const uint32_t koff = (kq >> 2) * 128 * 128 + (kq & 3) * 32;
                mma_tf32(tmem + kColG, sdesc_sw128(sbase + L::P + koff),
                         sdesc_sw128(sbase + L::P + 32768 + koff), idesc_tf32(128, 128), kq > 0);
            }
            mma_commit(bar_mma);
        }
        if (!wait_uniform(bar_mma, mma_parity, p.status)) { alive = false; break; }
        mma_parity ^= 1u;
        tc_fence_after_sync();

        // ---- phase 3: L_c -> LC scratch, L_k^T -> B_Y rows 64.., Qa^T -> B_Y rows 0..63
        {
            float *LC = reinterpret_cast<float *>(sm + L::AX);
            unsigned char *BY = sm + L::P + 32768;
            if (q >= 2) {
                const int t = 32 * (q - 2) + lane;  // Q rows of G sit in TMEM lanes 64..127
                float v[64];
                tmem_ld64(tmem + lane_off + kColG + 64 * hf, v);
                if (hf == 0) {  // L_c[t][s], s < t
#pragma unroll
                    for (int s0 = 0; s0 < 64; s0 += 4) {
                        float4 x;
                        x.x = (s0 < t) ? v[s0] : 0.f;
                        x.y = (s0 + 1 < t) ? v[s0 + 1] : 0.f;
                        x.z = (s0 + 2 < t) ? v[s0 + 2] : 0.f;
                        x.w = (s0 + 3 < t) ? v[s0 + 3] : 0.f;
                        *reinterpret_cast<float4 *>(LC + t * kLd + s0) = x;
                    }
                } else {  // B_Y[64 + s][t] = L_k[t][s]
#pragma unroll
                    for (int sidx = 0; sidx < 64; ++sidx)
                        *reinterpret_cast<uint32_t *>(BY + sw128_off(64 + sidx, t, 128)) =
                            to_tf32(sidx < t ? v[sidx] : 0.f);
                }
            } else {
                // Qa^T: B_Y[i][t] = kk[t][i] e^{g_{t-1}[i]}  (= kk * E[t-1] * eref, or kk at t = 0)
                const int lt = (warp & 1) * 32 + lane + 64 * (warp >> 2);  // warps 0,1,4,5 -> 0..127
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int i = lt & 63;
                    const int tc = (lt >> 6) + 2 * m;  // 0..15
                    const int tb = 4 * tc;
                    const float er = eref[i];
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = tb + e;
                        const float f = (t == 0) ? 1.f : Et[(t - 1) * 64 + i] * er;
                        x[e] = (t < lc) ? RawX::ld1(rkk, t, i) * f : 0.f;
                    }
                    st_tf32x4(BY + sw128_off(i, tb, 128), x[0], x[1], x[2], x[3]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- phase 4: T = (I + L_c)^{-1} in fp32 (TS), then T^T -> BX.
        // Diagonal 16x16 blocks by right-looking substitution in registers;
        // then the 32x32 halves T_A, T_B (T_10 = -T_11 L_10 T_00, likewise
        // T_32), then T_BA = -T_B (L_BA T_A).  Only lower-triangular entries of
        // TS are ever written or read; T^T takes zeros above the diagonal.
        {
            const float *LC = reinterpret_cast<const float *>(sm + L::AX);
            float *TS = reinterpret_cast<float *>(sm + L::P);
            float *XS = reinterpret_cast<float *>(sm + L::P + 64 * kLd * 4);  // 32 x 32 scratch
            if (tid < 64) {
                const int bb = tid >> 4, j = tid & 15, o = 16 * bb;
                float x[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) x[t] = (t == j) ? 1.f : 0.f;
#pragma unroll
                for (int u = 0; u < 15; ++u) {
#pragma unroll
                    for (int t = u + 1; t < 16; ++t) x[t] = fmaf(-LC[(o + t) * kLd + o + u], x[u], x[t]);
                }
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    if (t >= j) TS[(o + t) * kLd + o + j] = x[t];
            }
            __syncthreads();
            // Y1 = L_10 T_00 -> XS[0..255], Y3 = L_32 T_22 -> XS[256..511]  (T lower triangular:
            // entries above the diagonal are never written, so they are masked, not read as zero)
            {
                const int blk = tid >> 7, r = (tid >> 3) & 15, c0 = (tid & 7) * 2;
                const int o = 32 * blk;  // block (1,0) at rows 16.., cols 0..; block (3,2) at rows 48.., cols 32..
                float y0 = 0.f, y1 = 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float l = LC[(o + 16 + r) * kLd + o + u];
                    const float2 tt = *reinterpret_cast<const float2 *>(TS + (o + u) * kLd + o + c0);
                    y0 = fmaf(l, u >= c0 ? tt.x : 0.f, y0);
                    y1 = fmaf(l, u > c0 ? tt.y : 0.f, y1);
                }
                *reinterpret_cast<float2 *>(XS + blk * 256 + r * 16 + c0) = make_float2(y0, y1);
            }
            __syncthreads();
            // T_10 = -T_11 Y1, T_32 = -T_33 Y3
            {
                const int blk = tid >> 7, r = (tid >> 3) & 15, c0 = (tid & 7) * 2;
                const int o = 32 * blk;
                float t0 = 0.f, t1 = 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float a = u <= r ? TS[(o + 16 + r) * kLd + o + 16 + u] : 0.f;
                    const float2 y = *reinterpret_cast<const float2 *>(XS + blk * 256 + u * 16 + c0);
                    t0 = fmaf(a, y.x, t0);
                    t1 = fmaf(a, y.y, t1);
                }
                *reinterpret_cast<float2 *>(TS + (o + 16 + r) * kLd + o + c0) = make_float2(-t0, -t1);
            }
            __syncthreads();
            // Z = L_BA T_A (32 x 32) -> XS
            {
                const int r = tid >> 3, c0 = (tid & 7) * 4;
                float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const float l = LC[(32 + r) * kLd + u];
                    const float4 tA = *reinterpret_cast<const float4 *>(TS + u * kLd + c0);
                    z0 = fmaf(l, u >= c0 ? tA.x : 0.f, z0);
                    z1 = fmaf(l, u >= c0 + 1 ? tA.y : 0.f, z1);
                    z2 = fmaf(l, u >= c0 + 2 ? tA.z : 0.f, z2);
                    z3 = fmaf(l, u >= c0 + 3 ? tA.w : 0.f, z3);
                }
                *reinterpret_cast<float4 *>(XS + r * 32 + c0) = make_float4(z0, z1, z2, z3);
            }
            __syncthreads();
            // T_BA = -T_B Z
            {
                const int r = tid >> 3, c0 = (tid & 7) * 4;
                float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const float a = u <= r ? TS[(32 + r) * kLd + 32 + u] : 0.f;
                    const float4 z = *reinterpret_cast<const float4 *>(XS + u * 32 + c0);
                    t0 = fmaf(a, z.x, t0);
                    t1 = fmaf(a, z.y, t1);
                    t2 = fmaf(a, z.z, t2);
                    t3 = fmaf(a, z.w, t3);
                }
                *reinterpret_cast<float4 *>(TS + (32 + r) * kLd + c0) = make_float4(-t0, -t1, -t2, -t3);
            }
            __syncthreads();
            // T^T into BX: BX[n][k] = T[k][n] (zero above the diagonal)
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int n = tid & 63, kc = (tid >> 6) + 4 * m, k0 = 4 * kc;
                st_tf32x4(sm + L::BX + sw128_off(n, k0, 64), k0 >= n ? TS[k0 * kLd + n] : 0.f,
                          k0 + 1 >= n ? TS[(k0 + 1) * kLd + n] : 0.f, k0 + 2 >= n ? TS[(k0 + 2) * kLd + n] : 0.f,
                          k0 + 3 >= n ? TS[(k0 + 3) * kLd + n] : 0.f);
            }
            __syncthreads();  // LC (in AX) is dead from here on
        }

        // ---- phase 4b: A_X = [M_c ; Cb^T]; e^{g_C} saved for the state update
        {
            unsigned char *AXo = sm + L::AX;
            if (q < 2 && hf == 0) {
                const int t = 32 * q + lane;  // R rows of G sit in TMEM lanes 0..63
                float v[64];
                tmem_ld64(tmem + lane_off + kColG, v);
#pragma unroll
                for (int s0 = 0; s0 < 64; s0 += 4)
                    st_tf32x4(AXo + sw128_off(t, s0, 128), s0 <= t ? v[s0] : 0.f, s0 + 1 <= t ? v[s0 + 1] : 0.f,
                              s0 + 2 <= t ? v[s0 + 2] : 0.f, s0 + 3 <= t ? v[s0 + 3] : 0.f);
            } else {
                // Cb^T[i][s] = kk[s][i] a[s][i] e^{g_C[i] - g_s[i]} = c * E[63][i] / E[s][i]
                const int idx = tid - 64;  // warps 2..7 -> 0..191
                for (int e = idx; e < 1024; e += 192) {
                    const int i = e & 63, sc = e >> 6, s0 = 4 * sc;
                    const float e63 = Et[63 * 64 + i];
                    float x[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int ss = s0 + u;
                        x[u] = (ss < lc) ? RawX::ld1(rkk, ss, i) * RawX::ld1(ra, ss, i) * (e63 * rcp(Et[ss * 64 + i])) : 0.f;
                    }
                    st_tf32x4(AXo + sw128_off(64 + i, s0, 128), x[0], x[1], x[2], x[3]);
                }
                if (idx < 64) gC[idx] = Et[63 * 64 + idx] * eref[idx];
            }
        }
        sync_for_mma();

        // ---- MMA X: [M_c ; Cb^T] (128 x 64) x T -> TMEM X (128 x 64)
        if (tid == 0) {
#pragma unroll
            for (int kq = 0; kq < 8; ++kq) {
                mma_tf32(tmem + kColX, sdesc_sw128(sbase + L::AX + (kq >> 2) * 128 * 128 + (kq & 3) * 32),
                         sdesc_sw128(sbase + L::BX + (kq >> 2) * 64 * 128 + (kq & 3) * 32),
                         idesc_tf32(128, 64), kq > 0);
            }
            mma_commit(bar_mma);
        }
        if (!wait_uniform(bar_mma, mma_parity, p.status)) { alive = false; break; }
        mma_parity ^= 1u;
        tc_fence_after_sync();

        // ---- phase 5: A_Y = X (rows m, K = t) into P[0, 32K)
        {
            float v[32];
            tmem_ld32(tmem + lane_off + kColX + 32 * hf, v);
            const int m = 32 * q + lane;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                st_tf32x4(sm + L::P + sw128_off(m, 32 * hf + j, 128), v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
        sync_for_mma();

        // ---- MMA Y: [Mt ; Ct] x [Qa | L_k] -> TMEM Y (128 x 128)
        if (tid == 0) {
#pragma unroll
            for (int kq = 0; kq < 8; ++kq) {
                const uint32_t koff = (kq >> 2) * 128 * 128 + (kq & 3) * 32;
                mma_tf32(tmem + kColY, sdesc_sw128(sbase + L::P + koff),
                         sdesc_sw128(sbase + L::P + 32768 + koff), idesc_tf32(128, 128), kq > 0);
            }
            mma_commit(bar_mma);
        }
        if (!wait_uniform(bar_mma, mma_parity, p.status)) { alive = false; break; }
        mma_parity ^= 1u;
        tc_fence_after_sync();

        // ---- phase 6: A_chain (128 x K 128) in P
        //   rows t:    [ Ra - Mt Qa | M_k - Mt L_k ]      rows 64+i: [ -Ct Qa | Kb^T - Ct L_k ]
        {
            unsigned char *AC = sm + L::P;
            // pass 1: Ra (rows t, K 0..63) and Kb^T (rows 64+i, K 64..127) base values, fp32
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int task = tid + kThreads * m;
                const int t = task >> 4, i = (task & 15) * 4;
                const float valid = t < lc ? 1.f : 0.f;
                const float4 e = ld_f4(reinterpret_cast<unsigned char *>(Et + t * 64 + i));
                const float4 xr = RawX::ld4(rr, t, i);
                const float4 er = ld_f4(reinterpret_cast<unsigned char *>(eref + i));
                *reinterpret_cast<float4 *>(AC + sw128_off(t, i, 128)) =
                    make_float4(valid * xr.x * e.x * er.x, valid * xr.y * e.y * er.y,
                                valid * xr.z * e.z * er.z, valid * xr.w * e.w * er.w);
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int i = tid & 63, sc = (tid >> 6) + 4 * m, s0 = 4 * sc;
                const float e63 = Et[63 * 64 + i];
                float x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int ss = s0 + u;
                    x[u] = (ss < lc) ? RawX::ld1(rk, ss, i) * (e63 * rcp(Et[ss * 64 + i])) : 0.f;
                }
                *reinterpret_cast<float4 *>(AC + sw128_off(64 + i, 64 + s0, 128)) = make_float4(x[0], x[1], x[2], x[3]);
            }
            __syncthreads();
            // pass 2: combine with TMEM (Y, and M_k from G); each entry is rounded to tf32 once
            const int mrow = 32 * q + lane;
            float y[32], g[32];
            for (int half = 0; half < 2; ++half) {
                const int kb = 64 * hf + 32 * half;  // K columns of A_chain handled here
                tmem_ld32(tmem + lane_off + kColY + kb, y);
                if (q < 2 && hf == 1) tmem_ld32(tmem + lane_off + kColG + kb, g);  // R K^T block (M_k)
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    unsigned char *dst = AC + sw128_off(mrow, kb + j, 128);
                    float o4[4];
                    if ((q < 2 && hf == 0) || (q >= 2 && hf == 1)) {
                        const uint4 cur = *reinterpret_cast<const uint4 *>(dst);
                        o4[0] = __uint_as_float(cur.x) - y[j];
                        o4[1] = __uint_as_float(cur.y) - y[j + 1];
                        o4[2] = __uint_as_float(cur.z) - y[j + 2];
                        o4[3] = __uint_as_float(cur.w) - y[j + 3];
                    } else if (q < 2) {  // M_k - Mt L_k, M_k masked to s <= t
                        const int s0 = kb - 64 + j;
#pragma unroll
                        for (int u = 0; u < 4; ++u) o4[u] = (s0 + u <= mrow ? g[j + u] : 0.f) - y[j + u];
                    } else {  // -Ct Qa
#pragma unroll
                        for (int u = 0; u < 4; ++u) o4[u] = -y[j + u];
                    }
                    st_tf32x4(dst, o4[0], o4[1], o4[2], o4[3]);
                }
            }
        }
        sync_for_mma();

        // The raw tiles, E and AX are no longer read: fetch the next chunk now.
        if (tid == 0 && c + 1 < nchunks) issue_tma(c + 1);

        // ---- MMA chain: A_chain (128 x 128) x [S0 ; V] -> TMEM D (128 x 64)
        if (tid == 0) {
#pragma unroll
            for (int kq = 0; kq < 16; ++kq) {
                mma_tf32(tmem + kColD, sdesc_sw128(sbase + L::P + (kq >> 2) * 128 * 128 + (kq & 3) * 32),
                         sdesc_sw128(sbase + L::BC + (kq >> 2) * 64 * 128 + (kq & 3) * 32),
                         idesc_tf32(128, 64), kq > 0);
            }
            mma_commit(bar_mma);
        }
        if (!wait_uniform(bar_mma, mma_parity, p.status)) { alive = false; break; }
        mma_parity ^= 1u;
        tc_fence_after_sync();

        // ---- phase 7: outputs and the state update
        {
            float v[32];
            tmem_ld32(tmem + lane_off + kColD + 32 * hf, v);
            if (q < 2) {
                const int t = 32 * q + lane;
                if (t < lc) {
                    float4 *dst = reinterpret_cast<float4 *>(p.o + (t0 + t) * tok_stride + h * 64 + 32 * hf);
#pragma unroll
                    for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
            } else {
                const float decay = gC[srow];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = fmaf(decay, s[j], v[j]);
                    *reinterpret_cast<uint32_t *>(sm + L::BC + sw128_off(32 * hf + j, srow, 64)) = to_tf32(s[j]);
                }
            }
        }
        sync_for_mma();
    }

    if (alive && state_thread && p.final_state) {
        float4 *dst = reinterpret_cast<float4 *>(p.final_state + sslot + srow * 64 + 32 * hf);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool make_map(CUtensorMap *map, const void *base, bool bf16, int T_total, int H) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * 64, static_cast<cuuint64_t>(T_total)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 64 * esz};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename X>
cudaError_t launch_typed(const PrefillArgs &args, cudaStream_t stream) {
    using L = Layout<Raw<X>::kB>;
    const bool bf16 = Raw<X>::kB == 2;
    TensorMaps maps;
    if (!make_map(&maps.r, args.r, bf16, args.T_total, args.H) ||
        !make_map(&maps.k, args.k, bf16, args.T_total, args.H) ||
        !make_map(&maps.v, args.v, bf16, args.T_total, args.H) ||
        !make_map(&maps.kk, args.kk, bf16, args.T_total, args.H) ||
        !make_map(&maps.a, args.a, bf16, args.T_total, args.H) ||
        !make_map(&maps.w, args.w, false, args.T_total, args.H))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(wkv7_prefill_chunked_kernel<X>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const long long pairs = static_cast<long long>(args.num_seqs) * args.H;
    wkv7_prefill_chunked_kernel<X><<<static_cast<unsigned>(pairs), kThreads, L::kAlloc, stream>>>(args, maps);
    return cudaGetLastError();
}

}  // namespace

size_t prefill_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_prefill(const PrefillArgs &args, void *, size_t, cudaStream_t stream) {
    const long long pairs = static_cast<long long>(args.num_seqs) * args.H;
    if (pairs <= 0) return cudaSuccess;
    const size_t state_bytes = static_cast<size_t>(pairs) * 4096 * sizeof(float);
    if (args.T_total == 0) {  // every sequence is empty: final = initial (or zeros)
        if (!args.final_state) return cudaSuccess;
        if (!args.initial_state) return cudaMemsetAsync(args.final_state, 0, state_bytes, stream);
        if (args.initial_state == args.final_state) return cudaSuccess;
        return cudaMemcpyAsync(args.final_state, args.initial_state, state_bytes, cudaMemcpyDeviceToDevice, stream);
    }
    // bf16 inputs (the prefill format) take the chunked tensor-core kernel;
    // fp32 inputs take the exact token-serial kernel.
    if (args.x_dtype == WKV7_BF16) return launch_typed<__nv_bfloat16>(args, stream);
    return launch_prefill_scan(args, stream);
}

}  // namespace wkv7
