// Backward of the packed varlen prefill: the gradients of
//   L = <dO, o> + <dS_final, S_final>
// with respect to r, w, k, v, kk, a and the initial state, chunk by chunk.
//
// The recurrence (per head, S = [K, V]; Core AI model zoo, "Recurrent /
// linear-attention LLMs on Core AI", section 1):
//   z = kk^T S_old ;  S = diag(e^w) S_old - c z^T + k v^T (c = kk .* a) ;  o = S^T r
// is affine in S, so its adjoint G = dL/dS runs backwards with the transposed
// transition  G_old = diag(e^w) G - kk (c^T G)  plus r do^T at each read-out.
// The Pantheon RWKV-X page lists training (its forward with callbacks) among the
// Foundry engine's features, and the SwiftRWKV inference page notes that a
// fused kernel is opaque to autograd, so a training path needs the derivative
// written out.  The chunk algebra below is this library's own derivation,
// checked against the fp64 token-serial oracle.
//
// Per 64-token chunk with the local inclusive cumulative log-decay g_t, a
// reference rho = g_31 (decay factors stay within e^{+-32 |w|max}) and
//   R = r e^{g-rho}, Q = kk e^{g_{t-1}-rho}, K = k e^{rho-g}, Cm = c e^{rho-g},
//   Lc = tril_{-1}(Q Cm^T), Lk = tril_{-1}(Q K^T), Mc = tril_0(R Cm^T),
//   Mk = tril_0(R K^T), T = (I + Lc)^{-1}, S0' = e^{rho} S0, G' = e^{g_C-rho} Ghat:
//   forward :  Z = T (Q S0' + Lk V) ;  S_C = A S0 + F with
//              A = diag(e^{g_C-rho}) (I - Cm^T T Q) diag(e^{rho}),
//              F = diag(e^{g_C-rho}) (K^T - Cm^T T Lk) V
//   adjoint :  Ghat_prev = A^T Ghat + E,  E = diag(e^{rho}) (R^T - Q^T T^T Mc^T) dO
//   per chunk: U  = T^T (Cm G' + Mc^T dO)                  (u_t = G_t^T c_t)
//              dV = K G' + Mk^T dO - Lk^T U
//              dK = e^{rho-g} (V G'^T + triu_0(V dO^T) R - triu_1(V U^T) Q)
//              dC = -e^{rho-g} (Z G'^T + triu_0(Z dO^T) R - triu_1(Z U^T) Q)
//              dR = e^{g-rho} (dO S0'^T + tril_0(dO V^T) K - tril_0(dO Z^T) Cm)
//              dKr = -e^{g_{t-1}-rho} (U S0'^T + tril_{-1}(U V^T) K - tril_{-1}(U Z^T) Cm)
//              dkk = dKr + a dC,  da = kk dC
//   and, because the loss sees w only through the scaled operands and the
//   final state, dw_t = sum_{u>=t} (r dr - k dk - c dC)_u + sum_{u>t} (kk dKr)_u
//   + rowsum(Ghat .* S_C): a reverse cumulative sum inside the chunk plus a
//   carry from the chunk's end state.
//
// Launches (one stream, no host synchronisation):
//   1. chunk table: first chunk of every sequence (a prefix sum of ceil(len/64)).
//   2. summary (one CTA per chunk and head, all in parallel): A, F, E, and T and
//      the decay table g, which the gradient pass reads back instead of forming
//      them again.
//   3. chains (one CTA per sequence, head and direction): the states at every
//      chunk boundary forward, the adjoints at every chunk end backward.
//   4. gradients (one CTA per chunk and head, all in parallel).
// The summary and gradient passes run their products on the tensor cores
// (tcgen05, tf32 operands, fp32 accumulation in tensor memory); the chains
// multiply in fp32 on the CUDA cores (4 x 4 register tiles, operands in shared
// memory).  Only the two chains are sequential.  Whole 16 KB matrices (states,
// adjoints, T, g) move by single bulk copies and 64 x 64 outputs by one bulk copy
// per 256-byte row from staged shared-memory tiles, and both passes take the chunk's
// token rows (kk, k, a, r, v, dO) as 64-token TMA tiles, instead of per-thread row
// accesses (a warp's access touching 32 rows); only fp32 v rows and fp32 epilogue
// rows of the gradient pass, for which no shared memory is left, are loaded per thread.
#include <cuda_bf16.h>

#include <cstdint>

#include "sm103_ptx.cuh"
#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

using namespace ptx;

constexpr int kC = 64;            // tokens per chunk
constexpr int kLD = 68;           // shared-memory row stride in floats (16-B rows, staggered banks)
constexpr int kMat = kC * kLD;    // floats per 64 x 64 buffer
constexpr int kThreads = 256;
// The summary and gradient passes run 16 warps: a 128 x 64 operand row (TMEM lane) is split
// over four threads of kGW = 16 columns (kGroups = 4 column groups); the chains run 8 warps.
constexpr int kGradThreads = 512, kGW = 16, kGroups = 4;
constexpr size_t kMatBytes = (size_t)kMat * sizeof(float);
constexpr size_t kStateElems = (size_t)kN * kN;
constexpr size_t kChainSmem = 3 * kMatBytes;

struct BwdArgs {
    // 64-token tiles of kk, k, a, r for the TMA (128-byte swizzle: bf16 as one box of
    // 64 x 64, fp32 as two boxes of 64 x 32)
    CUtensorMap mkk, mk, ma, mr;
    CUtensorMap mv, mdo;  // v (like the above) and dO (fp32, two boxes of 64 x 32)
    int num_seqs;
    int H;
    const int32_t *cu;  // device cu_seqlens [num_seqs + 1]
    bool x_bf16;
    const void *r, *k, *v, *kk, *a;
    const float *w;
    const float *s0;   // nullable [num_seqs, H, 64, 64]
    const float *d_o;  // [T_total, H, 64]
    const float *dsf;  // nullable [num_seqs, H, 64, 64]
    float *dr, *dw, *dk, *dv, *dkk, *da;  // [T_total, H, 64]
    float *ds0;                           // nullable [num_seqs, H, 64, 64]
    int32_t *chunk_base;                  // [num_seqs + 1]
    float *Sck;  // [n_chunks + num_seqs, H, 64, 64] states at chunk boundaries
    float *Ack;  // [n_chunks, H, 64, 64]
    float *Fck;  // [n_chunks, H, 64, 64]
    float *Eck;  // [n_chunks, H, 64, 64]; E, then overwritten by the adjoint at the chunk end
    float *Tck;  // [n_chunks, H, 64, 64] T = (I + L_c)^{-1}, from the summary pass to the gradient pass
    float *Gck;  // [n_chunks, H, 64, 64] the cumulative log-decay g, likewise
    unsigned *status;  // device status word
};

// ---------------------------------------------------------------------------
// small helpers

__device__ __forceinline__ int tile_row() { return (threadIdx.x >> 4) * 4; }
__device__ __forceinline__ int tile_col() { return (threadIdx.x & 15) * 4; }

// acc[i][j] += (or -=) sum_{k in [k0, k1)} opA(m0 + i, k) * B[k][n0 + j], with
// opA(m, k) = A[m][k] (kTA = false) or A[k][m] (kTA = true); k0, k1 multiples of 4.
template <bool kTA, bool kNeg>
__device__ __forceinline__ void mm(float (&acc)[4][4], const float *__restrict__ A, const float *__restrict__ B,
                                   int k0, int k1) {
    const int m0 = tile_row(), n0 = tile_col();
#pragma unroll 2
    for (int k = k0; k < k1; k += 4) {
        float a[4][4];
        if (!kTA) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 x = *reinterpret_cast<const float4 *>(A + (m0 + i) * kLD + k);
                a[i][0] = x.x; a[i][1] = x.y; a[i][2] = x.z; a[i][3] = x.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 x = *reinterpret_cast<const float4 *>(A + (k + q) * kLD + m0);
                a[0][q] = x.x; a[1][q] = x.y; a[2][q] = x.z; a[3][q] = x.w;
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 b = *reinterpret_cast<const float4 *>(B + (k + q) * kLD + n0);
            const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float x = kNeg ? -a[i][q] : a[i][q];
                const float2 xx = make_float2(x, x);
                const float2 c01 = __ffma2_rn(xx, b01, make_float2(acc[i][0], acc[i][1]));
                const float2 c23 = __ffma2_rn(xx, b23, make_float2(acc[i][2], acc[i][3]));
                acc[i][0] = c01.x; acc[i][1] = c01.y;
                acc[i][2] = c23.x; acc[i][3] = c23.y;
            }
        }
    }
}

__device__ __forceinline__ void tile_store(float *dst, const float (&acc)[4][4]) {
    const int m0 = tile_row(), n0 = tile_col();
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(dst + (m0 + i) * kLD + n0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
}

// Triangular masks on (row, col): which entries a product keeps; the rest are zero.
enum Mask { kStrictLower, kLower, kUpper, kStrictUpper };
template <Mask M>
__device__ __forceinline__ bool keep(int row, int col) {
    if (M == kStrictLower) return col < row;
    if (M == kLower) return col <= row;
    if (M == kUpper) return col >= row;
    return col > row;
}
// Global [64][64] fp32 (row-major, 256 B rows) <-> shared [64][kLD]; nullptr loads zeros.
__device__ __forceinline__ void load_state(float *dst, const float *src) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int e = threadIdx.x + q * kThreads, row = e >> 4, c4 = (e & 15) * 4;
        const float4 x = src ? __ldg(reinterpret_cast<const float4 *>(src + row * kN + c4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(dst + row * kLD + c4) = x;
    }
}
__device__ __forceinline__ void store_state(float *dst, const float *src) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int e = threadIdx.x + q * kThreads, row = e >> 4, c4 = (e & 15) * 4;
        *reinterpret_cast<float4 *>(dst + row * kN + c4) = *reinterpret_cast<const float4 *>(src + row * kLD + c4);
    }
}

// The largest s with chunk_base[s] <= g (the sequence that owns global chunk g).
__device__ __forceinline__ int owner(const int32_t *cb, int num_seqs, int g) {
    int lo = 0, hi = num_seqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cb[mid] <= g) lo = mid; else hi = mid;
    }
    return lo;
}

struct Chunk {
    int seq, idx, tb, len;  // owning sequence, chunk index in it, first token, tokens (1..64)
};

__device__ __forceinline__ bool locate(const BwdArgs &p, int g, Chunk &c) {
    if (g >= p.chunk_base[p.num_seqs]) return false;
    c.seq = owner(p.chunk_base, p.num_seqs, g);
    c.idx = g - p.chunk_base[c.seq];
    c.tb = p.cu[c.seq] + c.idx * kC;
    c.len = min(kC, p.cu[c.seq + 1] - c.tb);
    return true;
}

// T = (I + Lc)^{-1} for the strictly lower Lc: the four 16 x 16 diagonal blocks by
// forward substitution (one thread of warps 2 and 3 per column: warps 0 and 1 may still
// be issuing products; the other threads meanwhile zero the six blocks above them), then
// the blocks below them by
// T_IJ = -T_II sum_{K=J}^{I-1} Lc_IK T_KJ, one block diagonal at a time, each thread
// taking four consecutive columns of a row (16-byte loads of Lc and T rows, four
// independent sums).  tmp holds at least 3 * 256 floats.  NT threads.  Ends with a barrier.
template <int NT>
__device__ void unit_lower_inverse(const float *Lc, float *T, float *tmp) {
    const int tid = threadIdx.x;
    if (tid >= 64 && tid < 128) {
        const int o = ((tid - 64) >> 4) * 16, jj = tid & 15;
        float x[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            float acc = t == jj ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < t; ++s) acc = fmaf(-Lc[(o + t) * kLD + o + s], x[s], acc);
            x[t] = acc;
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) T[(o + t) * kLD + o + jj] = x[t];
    } else {
        for (int e = tid < 64 ? tid : tid - 64; e < 6 * 64; e += NT - 64) {  // blocks (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
            const int blk = e >> 6, row = (e >> 2) & 15, c4 = (e & 3) * 4;
            const int I = blk < 3 ? 0 : (blk < 5 ? 1 : 2), J = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            *reinterpret_cast<float4 *>(T + (I * 16 + row) * kLD + J * 16 + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();
    for (int d = 1; d < 4; ++d) {
        const int np = 4 - d;
        for (int e = tid; e < np * 64; e += NT) {  // tmp_J = sum_{K=J}^{I-1} Lc_IK T_KJ, row rr, columns c4..
            const int J = e >> 6, rr = (e >> 2) & 15, c4 = (e & 3) * 4, I = J + d;
            const float *lrow = Lc + (I * 16 + rr) * kLD;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int kb = J; kb < I; ++kb) {
#pragma unroll
                for (int q4 = 0; q4 < 16; q4 += 4) {
                    const float4 l = *reinterpret_cast<const float4 *>(lrow + kb * 16 + q4);
                    const float lq[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const float4 tv = *reinterpret_cast<const float4 *>(T + (kb * 16 + q4 + qq) * kLD + J * 16 + c4);
                        acc.x = fmaf(lq[qq], tv.x, acc.x);
                        acc.y = fmaf(lq[qq], tv.y, acc.y);
                        acc.z = fmaf(lq[qq], tv.z, acc.z);
                        acc.w = fmaf(lq[qq], tv.w, acc.w);
                    }
                }
            }
            *reinterpret_cast<float4 *>(tmp + (J << 8) + rr * 16 + c4) = acc;
        }
        __syncthreads();
        for (int e = tid; e < np * 64; e += NT) {  // T_IJ = -T_II tmp_J, row rr, columns c4..
            const int J = e >> 6, rr = (e >> 2) & 15, c4 = (e & 3) * 4, I = J + d;
            const float *trow = T + (I * 16 + rr) * kLD + I * 16;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q4 = 0; q4 < 16; q4 += 4) {
                const float4 tr = *reinterpret_cast<const float4 *>(trow + q4);
                const float tq[4] = {tr.x, tr.y, tr.z, tr.w};
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const float4 m = *reinterpret_cast<const float4 *>(tmp + (J << 8) + (q4 + qq) * 16 + c4);
                    acc.x = fmaf(tq[qq], m.x, acc.x);
                    acc.y = fmaf(tq[qq], m.y, acc.y);
                    acc.z = fmaf(tq[qq], m.z, acc.z);
                    acc.w = fmaf(tq[qq], m.w, acc.w);
                }
            }
            *reinterpret_cast<float4 *>(T + (I * 16 + rr) * kLD + J * 16 + c4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// 1. chunk table: chunk_base[s] = sum_{s' < s} ceil(len_s' / 64).  A malformed
// cu_seqlens (not starting at 0, decreasing, or not ending at T_total) is
// reported and leaves a table with no chunks, so no later launch touches a token.

__global__ void __launch_bounds__(1024) bwd_chunk_table_kernel(const int32_t *cu, int num_seqs, int T_total,
                                                               int32_t *cb, unsigned *status) {
    __shared__ int32_t part[1024];
    __shared__ int bad;
    const int tid = threadIdx.x;
    if (tid == 0) bad = (cu[0] != 0 || cu[num_seqs] != T_total) ? 1 : 0;
    __syncthreads();
    const int per = (num_seqs + 1023) / 1024;
    const int s0 = tid * per, s1 = min(num_seqs, s0 + per);
    int32_t sum = 0;
    for (int s = s0; s < s1; ++s) {
        const int len = cu[s + 1] - cu[s];
        if (len < 0) bad = 1;
        else sum += (len + kC - 1) / kC;
    }
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        int32_t run = 0;
        for (int i = 0; i < 1024; ++i) {
            const int32_t v = part[i];
            part[i] = run;
            run += v;
        }
        cb[num_seqs] = bad ? 0 : run;
        if (bad) report(status, kDevBadSeqlens);
    }
    __syncthreads();
    int32_t run = bad ? 0 : part[tid];
    for (int s = s0; s < s1; ++s) {
        cb[s] = run;
        if (!bad) run += (cu[s + 1] - cu[s] + kC - 1) / kC;
    }
}

// ---------------------------------------------------------------------------
// tensor-core helpers shared by the summary and gradient passes

namespace tcg {
// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t kBG = 0;           // [Cm; K; R; Q], 256 rows x K 64 (64 KB), stage 1
constexpr uint32_t kBY = 0;           // [S0'^T | V^c] 64 x 128 (32 KB), stage 2; then Y^c, Y2^c; then B_P
constexpr uint32_t kBF3 = 32768;      // [G'^T | dO^c | U^c] 64 x 192 (48 KB), stages 2 and 4
constexpr uint32_t kBF1 = 81920;      // [G' | R^c | Q^c] 64 x 192 (48 KB), stage 6
constexpr uint32_t kBF2 = 131072;     // [S0' | K^c | Cm^c] 64 x 192 (48 KB), stage 6
constexpr uint32_t kStage = 81920;    // epilogue (B_F1, B_F2 done): fp32 64 x 68 tiles of da, dkk, dk, dr, dw
constexpr uint32_t kDv = 32768;       // after stage 4 (B_F3 done) to stage 6: fp32 64 x 68 tile of dV
constexpr uint32_t kPlain0 = 180224;  // fp32 64 x 68: the cumulative decay, then T; then (with kPlain1) B_Pt
constexpr uint32_t kPlain1 = 197632;  // fp32 64 x 68: Lc
constexpr uint32_t kVec = 215040;     // rho[64], gC[64], carry parts [4][64]
constexpr uint32_t kBar = 216576;     // mbarrier, TMEM base slot; mbarriers of the states, T, the decay table,
                                      // the raw tiles, the v and dO tiles, the epilogue's raw tiles
// the bf16 v tile by TMA (an fp32 one does not fit: fp32 v rows are loaded per thread); the
// dO tile goes to the second plain buffer (free until B_Pt), the epilogue's raw tiles (bf16)
// to both plain buffers (free after stage 5)
constexpr uint32_t kVt = 217088;
constexpr uint32_t kBytes = kVt + 8192;
// S0, Ghat and S_C (16 KB each, unpadded) arrive by bulk copies at the CTA's start and are
// read in the B-tile step: places no operand uses before then (B_F3's U^c part, B_F1's and
// B_F2's first K = 64, written in that step after a barrier)
constexpr uint32_t kSt0 = 65536, kSt1 = 81920, kSt2 = 131072;
constexpr uint32_t kAlloc = kBytes + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kMaxPolls = 1u << 24;
constexpr uint32_t kAtom64 = 64 * 128, kAtom128 = 128 * 128, kAtom256 = 256 * 128;
static_assert(kStage + 5 * kMatBytes <= kPlain0, "gradient staging tiles overlap the plain buffers");
static_assert(kDv >= kBF3 && kDv + kMatBytes <= kBF1, "the dV tile lies outside B_F3");
static_assert(kPlain1 == kPlain0 + kMatBytes && kPlain1 + kMatBytes <= kVec, "B_Pt spans both plain buffers");
static_assert(kVt % 1024 == 0 && kVt >= kBar + 64 && kPlain0 % 1024 == 0 && kPlain1 % 1024 == 0 &&
                  kPlain1 + 16384 <= kVec && kPlain0 + 4 * 8192 <= kVec,
              "TMA tiles: 1024-byte aligned, inside their regions");
static_assert(kSt0 >= kBG + 256 * 256 && kSt0 + 16384 <= kBF1 && kSt1 == kBF1 && kSt2 == kBF2,
              "a staged state overlaps an operand in use before the B-tile step");
static_assert((kLD * sizeof(float)) % 16 == 0, "staged rows must start on 16-byte boundaries for the bulk stores");
}  // namespace tcg

__device__ __forceinline__ uint32_t tf32r(float x) { return __float_as_uint(x) + 0x1000u; }

// W (16 or 32) consecutive values of one packed token row, widened to fp32.
template <int W>
__device__ __forceinline__ void load_row(float (&v)[W], const void *src, bool bf16, size_t off) {
    if (bf16) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(src) + off);
#pragma unroll
        for (int q = 0; q < W / 8; ++q) {
            const uint4 u = __ldg(p + q);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[8 * q + 2 * e] = __uint_as_float(w4[e] << 16);
                v[8 * q + 2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
            }
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + off);
#pragma unroll
        for (int q = 0; q < W / 4; ++q) {
            const float4 x = __ldg(p + q);
            v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
        }
    }
}
template <int W>
__device__ __forceinline__ void zero_row(float (&v)[W]) {
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = 0.f;
}
// W values of row `row` of a plain [64][kLD] buffer from column c0 (float4 reads).
template <int W>
__device__ __forceinline__ void plain_row(float (&v)[W], const float *buf, int row, int c0) {
#pragma unroll
    for (int q = 0; q < W / 4; ++q) {
        const float4 x = *reinterpret_cast<const float4 *>(buf + row * kLD + c0 + 4 * q);
        v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
}
template <int W>
__device__ __forceinline__ void plain_row_store(float *buf, int row, int c0, const float (&v)[W]) {
#pragma unroll
    for (int q = 0; q < W / 4; ++q)
        *reinterpret_cast<float4 *>(buf + row * kLD + c0 + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
// Row `row`, K = kofs .. kofs + W - 1 of a K-major 128B-swizzled tile with `rows` rows.
template <int W>
__device__ __forceinline__ void b_row(unsigned char *tile, int rows, int row, int kofs, const float (&v)[W]) {
#pragma unroll
    for (int q = 0; q < W / 4; ++q)
        *reinterpret_cast<uint4 *>(tile + sw128_off(row, kofs + 4 * q, rows)) =
            make_uint4(tf32r(v[4 * q]), tf32r(v[4 * q + 1]), tf32r(v[4 * q + 2]), tf32r(v[4 * q + 3]));
}
// Column k of the tile, rows n0 .. n0 + W - 1 (a transposed store of this thread's row).
template <int W>
__device__ __forceinline__ void b_col(unsigned char *tile, int rows, int k, int n0, const float (&v)[W]) {
#pragma unroll
    for (int c = 0; c < W; ++c) *reinterpret_cast<uint32_t *>(tile + sw128_off(n0 + c, k, rows)) = tf32r(v[c]);
}
// This thread's TMEM lane, W columns from taddr: tf32 operand values / raw reads.
template <int W>
__device__ __forceinline__ void a_row(uint32_t taddr, const float (&v)[W]) {
    uint32_t r[W];
#pragma unroll
    for (int i = 0; i < W; ++i) r[i] = tf32r(v[i]);
    if constexpr (W == 32) tmem_st32u(taddr, r);
    else tmem_st16(taddr, r);
}
// Two (three) 16-column loads of this thread's TMEM lane with one wait, in one asm
// statement so that no use of the outputs is scheduled before the wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float (&va)[16], float (&vb)[16]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[16 + i]);
    }
}
__device__ __forceinline__ void tmem_ld16x3(uint32_t ta, uint32_t tb, uint32_t tc, float (&va)[16], float (&vb)[16],
                                            float (&vc)[16]) {
    uint32_t r[48];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%48];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%49];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47}, [%50];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
        : "r"(ta), "r"(tb), "r"(tc)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[16 + i]);
        vc[i] = __uint_as_float(r[32 + i]);
    }
}
// A 16-column store without its wait (tmem_wait_st before an MMA reads the columns).
__device__ __forceinline__ void tmem_st16_issue(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// As a_row for 16 columns, without the wait (tmem_wait_st before an MMA reads them).
__device__ __forceinline__ void a_row_issue(uint32_t taddr, const float (&v)[16]) {
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = tf32r(v[i]);
    tmem_st16_issue(taddr, r);
}
template <int W>
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const uint32_t (&r)[W]) {
    if constexpr (W == 32) tmem_st32u(taddr, r);
    else tmem_st16(taddr, r);
}
template <int W>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, float (&v)[W]) {
    if constexpr (W == 32) tmem_ld32(taddr, v);
    else tmem_ld16(taddr, v);
}

// Keep entries of row `row`, columns c0 .. c0 + W - 1, whose column passes the mask; optionally negate.
template <Mask M, bool kNegate, int W>
__device__ __forceinline__ void mask_row(float (&v)[W], int row, int c0) {
#pragma unroll
    for (int c = 0; c < W; ++c) {
        const float x = kNegate ? -v[c] : v[c];
        v[c] = keep<M>(row, c0 + c) ? x : 0.f;
    }
}

// D[dcol..] = A[tmem acol..] x B^T with B a K-major tile at bsaddr (atom_bytes per 32 K).
__device__ __forceinline__ void mma_group(uint32_t tmem, uint32_t dcol, uint32_t acol, uint32_t bsaddr,
                                          uint32_t atom_bytes, int n, int k) {
    const uint32_t idesc = idesc_tf32(128, n);
    for (int kq = 0; kq < k / 8; ++kq)
        mma_tf32_tmem_a(tmem + dcol, tmem + acol + 8 * kq,
                        sdesc_sw128(bsaddr + (kq >> 2) * atom_bytes + (kq & 3) * 32), idesc, kq > 0 ? 1u : 0u);
}

// As mma_group, with the A operand negated and/or accumulating onto D from the first step.
__device__ __forceinline__ void mma_group_acc(uint32_t tmem, uint32_t dcol, uint32_t acol, uint32_t bsaddr,
                                              uint32_t atom_bytes, int n, int k, bool negate, bool accumulate) {
    const uint32_t idesc = idesc_tf32(128, n) | (negate ? kIdescNegateA : 0u);
    for (int kq = 0; kq < k / 8; ++kq)
        mma_tf32_tmem_a(tmem + dcol, tmem + acol + 8 * kq,
                        sdesc_sw128(bsaddr + (kq >> 2) * atom_bytes + (kq & 3) * 32), idesc,
                        (accumulate || kq > 0) ? 1u : 0u);
}

// The products of a stage are issued by two threads, lane 0 of warps 0 and 1 (issuer 0
// and 1), each taking its own independent groups (a group and whatever accumulates onto
// its D stay with one issuer, so they keep their order): an issuing thread is held for
// ~70 cycles per instruction, and every barrier after it waits for its warp.
constexpr int kIssuers = 2;
__device__ __forceinline__ int issuer_id() {
    return (threadIdx.x & 31) == 0 && threadIdx.x < 32 * kIssuers ? static_cast<int>(threadIdx.x >> 5) : -1;
}

// Operands written -> the issuers issue, without a commit: the products run while the
// threads go on, and the next mma_stage's commits and wait cover them too.
template <class F>
__device__ __forceinline__ void mma_issue(F issue) {
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    const int who = issuer_id();
    if (who >= 0) {
        tc_fence_after_sync();
        issue(who);
    }
}

// Operands written -> the issuers issue and each commits (the mbarrier counts kIssuers
// arrivals) -> every thread waits (bounded).  The outcome is uniform over the CTA; false
// after a timeout (reported).
template <class F>
__device__ __forceinline__ bool mma_stage(uint32_t bar, uint32_t &phase, unsigned *status, F issue) {
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    const int who = issuer_id();
    if (who >= 0) {
        tc_fence_after_sync();
        issue(who);
        mma_commit(bar);
    }
    const bool ok = mbar_wait_bounded(bar, phase, tcg::kMaxPolls);
    phase ^= 1u;
    const int all_ok = __syncthreads_and(ok ? 1 : 0);
    tc_fence_after_sync();
    if (!all_ok && threadIdx.x == 0) report(status, kDevTimeout);
    return all_ok != 0;
}

// This thread's 4096 / NT values of w for the cumulative sum (row tid / (NT / 64), the
// consecutive channels from (tid mod (NT / 64)) x 4096 / NT) with NT threads.
template <int NT>
__device__ __forceinline__ void load_w(float (&x)[4096 / NT], const BwdArgs &p, const Chunk &c, int h) {
    constexpr int kPer = 4096 / NT;
    const int t = threadIdx.x / (NT / 64), cc = (threadIdx.x % (NT / 64)) * kPer;
    const bool valid = t < c.len;
    if (valid) {
        const float4 *src = reinterpret_cast<const float4 *>(p.w + ((size_t)(c.tb + t) * p.H + h) * kN + cc);
#pragma unroll
        for (int q = 0; q < kPer / 4; ++q) {
            const float4 w4 = __ldg(src + q);
            x[4 * q] = w4.x; x[4 * q + 1] = w4.y; x[4 * q + 2] = w4.z; x[4 * q + 3] = w4.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < kPer; ++j) x[j] = 0.f;
    }
    float wmin = 0.f;
#pragma unroll
    for (int j = 0; j < kPer; ++j) wmin = fminf(wmin, x[j]);
    if (valid && wmin < kMinLogDecay) report(p.status, kDevDomain);  // outside the domain: reported
}

// Inclusive cumulative sum of w over the chunk into Gm ([64][kLD]) from the values
// of load_w, with NT threads (NT / 64 row segments of 4096 / NT rows); scratch: NT / 64
// rows of kLD.  Ends with a barrier.
template <int NT>
__device__ void decay_cumsum_from(const float (&x)[4096 / NT], float *Gm, float *scratch) {
    constexpr int kPer = 4096 / NT;
    float *dst = Gm + (threadIdx.x / (NT / 64)) * kLD + (threadIdx.x % (NT / 64)) * kPer;
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q)
        *reinterpret_cast<float4 *>(dst + 4 * q) = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    __syncthreads();
    const int ch = threadIdx.x & 63, qt = threadIdx.x >> 6;
    float run = 0.f;
    float part[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        run += Gm[(qt * kPer + u) * kLD + ch];
        part[u] = run;
    }
    scratch[qt * kLD + ch] = run;
    __syncthreads();
    float base = 0.f;
    for (int q = 0; q < qt; ++q) base += scratch[q * kLD + ch];
#pragma unroll
    for (int u = 0; u < kPer; ++u) Gm[(qt * kPer + u) * kLD + ch] = part[u] + base;
    __syncthreads();
}

template <int NT>
__device__ void decay_cumsum(const BwdArgs &p, const Chunk &c, int h, float *Gm, float *scratch) {
    float x[4096 / NT];
    load_w<NT>(x, p, c, h);
    decay_cumsum_from<NT>(x, Gm, scratch);
}

// Row `row`, columns c0 .. c0 + 15 of an unpadded 64 x 64 fp32 matrix in shared memory.
// A warp's 32 rows start in one bank, so each lane reads its four 16-byte words in an
// order rotated by its row (four bank groups per access instead of one).
__device__ __forceinline__ void staged_row16(float (&v)[16], const float *m, int row, int c0) {
    const int r = row & 3;
    float4 w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = *reinterpret_cast<const float4 *>(m + row * kN + c0 + 4 * ((k + r) & 3));
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // word q was read at step (q - r) mod 4
        const int k = (q - r) & 3;
        const float4 x = k == 0 ? w[0] : k == 1 ? w[1] : k == 2 ? w[2] : w[3];
        v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
}

// The chunk's raw tiles of kk, k, a, r (in that order, kRawTile apart from dst) by TMA,
// completion on `bar`; rows past T_total arrive as zeros, rows of the next sequence
// are loaded and not used.  One thread.
__device__ __forceinline__ void issue_raw_tiles(const BwdArgs &p, const Chunk &c, int h, uint32_t dst, uint32_t bar) {
    const uint32_t tile = p.x_bf16 ? 8192u : 16384u;
    mbar_arrive_expect_tx(bar, 4 * tile);
    const CUtensorMap *maps[4] = {&p.mkk, &p.mk, &p.ma, &p.mr};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        tma_load_2d(dst + i * tile, maps[i], h * 64, c.tb, bar);
        if (!p.x_bf16) tma_load_2d(dst + i * tile + 8192, maps[i], h * 64 + 32, c.tb, bar);
    }
}
// 16 values of row t from channel c0 of a raw tile (128-byte rows whose 16-byte chunks
// are XOR-swizzled by t mod 8), widened from bf16.
__device__ __forceinline__ void raw_row16(float (&v)[16], const unsigned char *tile, bool bf16, int t, int c0) {
    if (bf16) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int chunk = (c0 >> 3) + q;
            const uint4 u = *reinterpret_cast<const uint4 *>(tile + t * 128 + ((chunk ^ (t & 7)) << 4));
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[8 * q + 2 * e] = __uint_as_float(w4[e] << 16);
                v[8 * q + 2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
            }
        }
    } else {
        const unsigned char *box = tile + (c0 >> 5) * 8192;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int chunk = ((c0 & 31) >> 2) + q;
            const float4 x = *reinterpret_cast<const float4 *>(box + t * 128 + ((chunk ^ (t & 7)) << 4));
            v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
        }
    }
}
// The chunk's dO tile (two fp32 boxes) at dst_o and, with_v, its v tile at dst_v, by TMA,
// completion on `bar`.  One thread.
__device__ __forceinline__ void issue_vdo_tiles(const BwdArgs &p, const Chunk &c, int h, uint32_t dst_v, uint32_t dst_o,
                                                uint32_t bar, bool with_v) {
    const uint32_t vbytes = with_v ? (p.x_bf16 ? 8192u : 16384u) : 0u;
    mbar_arrive_expect_tx(bar, vbytes + 16384u);
    if (with_v) {
        tma_load_2d(dst_v, &p.mv, h * 64, c.tb, bar);
        if (!p.x_bf16) tma_load_2d(dst_v + 8192, &p.mv, h * 64 + 32, c.tb, bar);
    }
    tma_load_2d(dst_o, &p.mdo, h * 64, c.tb, bar);
    tma_load_2d(dst_o + 8192, &p.mdo, h * 64 + 32, c.tb, bar);
}
// This thread's start rows from the raw tiles: top kk, k; bottom kk, a, r (zeros past the chunk).
__device__ __forceinline__ void raw_start_rows(float (&kk)[16], float (&ra)[16], float (&rb)[16],
                                               const unsigned char *tiles, bool bf16, bool top, bool valid, int t,
                                               int c0) {
    const int tile = bf16 ? 8192 : 16384;
    if (valid) {
        raw_row16(kk, tiles, bf16, t, c0);
        raw_row16(ra, tiles + (top ? 1 : 2) * tile, bf16, t, c0);
        if (!top) raw_row16(rb, tiles + 3 * tile, bf16, t, c0);
    } else {
        zero_row(kk); zero_row(ra); zero_row(rb);
    }
}

// ---------------------------------------------------------------------------
// 2. per-chunk summary on the tensor cores: A, F (forward transition) and E
// (adjoint input).  Their products contract over tokens, so their left
// operands have channels for rows: those come from identity products
// ([I 0; 0 I] x [X | Y]^T puts X^T in the top lanes and Y^T in the bottom ones)
// and from products whose own left operand already has channels for rows.
// Stages:
//   1  G1 = [Q; Cm] x [Cm; K; R]^T -> Lc, Lk (top), Mc^T (bottom);
//      [Cm^T; Q^T] and [K^T; R^T] by identity products
//   2  Lk V (top), Mc^T dO (bottom); W1 = Cm^T T (top), W2 = Q^T T^T (bottom)
//   3  F* = K^T V - W1 (Lk V) (top), E* = R^T dO - W2 (Mc^T dO) (bottom), A* = W1 Q (top)
// then A = diag(e^{gC-rho})(I - A*)diag(e^{rho}), F = diag(e^{gC-rho}) F*, E = diag(e^{rho}) E*.

namespace tcs {
constexpr uint32_t kBG = 0;           // [Cm; K; R; Q], 256 rows x K 64 (64 KB), stage 1; then stage-2 tiles
constexpr uint32_t kBVc = 0;          // V^c (16 KB), stages 2 and 3
constexpr uint32_t kBdOc = 16384;     // dO^c (16 KB), stages 2 and 3
constexpr uint32_t kBTt = 32768;      // rows t: T[s][t] (16 KB), stage 2
constexpr uint32_t kBTn = 49152;      // rows t: T[t][s] (16 KB), stage 2
constexpr uint32_t kBT1 = 65536;      // [Cm | Q] 64 x K 128 (32 KB), stage 1; then (Lk V)^c, (Mc^T dO)^c
constexpr uint32_t kBT2 = 98304;      // [K | R] 64 x K 128 (32 KB), stage 1
constexpr uint32_t kBQc = 131072;     // Q^c (16 KB), stage 3
constexpr uint32_t kPlain0 = 147456;  // fp32 64 x 68: the cumulative decay, then T
constexpr uint32_t kPlain1 = 164864;  // fp32 64 x 68: Lc
constexpr uint32_t kStage = 0;        // after stage 3: fp32 64 x 68 tiles of F, A, E for the bulk row stores
static_assert(kStage + 3 * kMatBytes <= kPlain0, "output staging tiles overlap the plain buffers");
constexpr uint32_t kVec = 182272;     // rho[64], gC[64]
constexpr uint32_t kBar = 182784;     // mbarrier, TMEM base slot, the raw tiles' and the v, dO tiles' mbarriers
// v and dO tiles by TMA (v: 8 KB bf16 or 16 KB fp32; dO 16 KB), 1024-byte aligned for the swizzle
constexpr uint32_t kVt = 183296, kdOt = kVt + 16384;
constexpr uint32_t kBytes = kdOt + 16384;
constexpr uint32_t kAlloc = kBytes + 1024;
}  // namespace tcs

__global__ void __launch_bounds__(kGradThreads, 1) bwd_summary_tc_kernel(const __grid_constant__ BwdArgs p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Chunk c;
    if (!locate(p, blockIdx.x, c)) return;
    const int h = blockIdx.y;
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hh = warp >> 2;
    const int L = 32 * quad + lane, t = L & 63, c0 = kGW * hh;
    const bool top = L < 64;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    float *rho = reinterpret_cast<float *>(sm + tcs::kVec), *gC = rho + 64;
    float *P0 = reinterpret_cast<float *>(sm + tcs::kPlain0), *P1p = reinterpret_cast<float *>(sm + tcs::kPlain1);
    const uint32_t bar = sbase + tcs::kBar, bar_x = sbase + tcs::kBar + 16, bar_v = sbase + tcs::kBar + 24;
    const size_t cidx = ((size_t)blockIdx.x * p.H + h) * kStateElems;
    const bool row_valid = t < c.len;

    if (tid == 0) {
        mbar_init(bar, kIssuers);
        mbar_init(bar_x, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
        issue_raw_tiles(p, c, h, sbase + tcs::kBG, bar_x);  // B_G's space, written after they are read
        issue_vdo_tiles(p, c, h, sbase + tcs::kVt, sbase + tcs::kdOt, bar_v, true);
    }
    if (warp == 0) tmem_alloc(sbase + tcs::kBar + 8, tcg::kTmemCols);
    decay_cumsum<kGradThreads>(p, c, h, P0, P1p);  // (its barriers publish bar_x's initialisation)
    float kk[kGW], ra[kGW], rb[kGW];  // top: kk, k; bottom: kk, a, r
    if (!mbar_wait_bounded(bar_x, 0, tcg::kMaxPolls)) report(p.status, kDevTimeout);
    raw_start_rows(kk, ra, rb, sm + tcs::kBG, p.x_bf16, top, row_valid, t, c0);
    if (tid < 64) {
        rho[tid] = P0[31 * kLD + tid];
        gC[tid] = P0[63 * kLD + tid];
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // the decay table for the gradient pass, one 256-byte bulk copy per row (read before
    // the inverse writes T over it)
    if (tid < kC)
        bulk_store(p.Gck + cidx + tid * kN, sbase + tcs::kPlain0 + (uint32_t)(tid * kLD * sizeof(float)),
                   kN * sizeof(float));
    bulk_commit();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + tcs::kBar + 8);
    const uint32_t tl = tmem + lane_off + c0;
    uint32_t phase = 0;
    bool ok = true;
    float v[kGW], x[kGW];

    // ---- scaled operands (top rows Q, K; bottom rows Cm, R) and the identity [I 0; 0 I] at 256..383
    {
        float g[kGW], gx[kGW];
        plain_row(g, P0, t, c0);
        if (t > 0) plain_row(gx, P0, t - 1, c0); else zero_row(gx);
        if (top) {
#pragma unroll
            for (int i = 0; i < kGW; ++i) {
                const float rh = rho[c0 + i];
                v[i] = kk[i] * __expf(gx[i] - rh);  // Q
                x[i] = ra[i] * __expf(rh - g[i]);   // K
            }
            a_row(tl + 0, v);
            b_row(sm + tcs::kBG, 256, 64 + t, c0, x);
            b_row(sm + tcs::kBG, 256, 192 + t, c0, v);
            b_row(sm + tcs::kBT1, 64, t, 64 + c0, v);
            b_row(sm + tcs::kBT2, 64, t, c0, x);
            b_col(sm + tcs::kBQc, 64, t, c0, v);
        } else {
#pragma unroll
            for (int i = 0; i < kGW; ++i) {
                const float rh = rho[c0 + i];
                v[i] = kk[i] * ra[i] * __expf(rh - g[i]);  // Cm
                x[i] = rb[i] * __expf(g[i] - rh);          // R
            }
            a_row(tl + 0, v);
            b_row(sm + tcs::kBG, 256, t, c0, v);
            b_row(sm + tcs::kBG, 256, 128 + t, c0, x);
            b_row(sm + tcs::kBT1, 64, t, c0, v);
            b_row(sm + tcs::kBT2, 64, t, 64 + c0, x);
        }
        uint32_t id[kGW];
#pragma unroll
        for (int i = 0; i < kGW; ++i) id[i] = (top && c0 + i == t) ? 0x3f800000u : 0u;
        tmem_st_row(tl + 256, id);
#pragma unroll
        for (int i = 0; i < kGW; ++i) id[i] = (!top && c0 + i == t) ? 0x3f800000u : 0u;
        tmem_st_row(tl + 320, id);
    }
    ok = mma_stage(bar, phase, p.status, [&](int who) {
        if (who == 0) {
            mma_group(tmem, 64, 0, sbase + tcs::kBG, tcg::kAtom256, 192, 64);     // G1
            mma_group(tmem, 384, 256, sbase + tcs::kBT1, tcg::kAtom64, 64, 128);  // [Cm^T; Q^T]
        } else {
            mma_group(tmem, 448, 256, sbase + tcs::kBT2, tcg::kAtom64, 64, 128);  // [K^T; R^T]
        }
    });

    if (ok) {
        // ---- Lc -> plain; A_L = [Lk (top); Mc^T (bottom)] at 64
        if (top) {
            tmem_ld_row(tl + 64, v);
            mask_row<kStrictLower, false>(v, t, c0);
            plain_row_store(P1p, t, c0, v);
            tmem_ld_row(tl + 128, v);
            mask_row<kStrictLower, false>(v, t, c0);
            a_row(tl + 64, v);
        } else {
            tmem_ld_row(tl + 192, v);
            mask_row<kUpper, false>(v, t, c0);
            a_row(tl + 64, v);
            if (!mbar_wait_bounded(bar_v, 0, tcg::kMaxPolls)) report(p.status, kDevTimeout);
            if (row_valid) {  // this row of v and dO
                raw_row16(kk, sm + tcs::kVt, p.x_bf16, t, c0);
                raw_row16(ra, sm + tcs::kdOt, false, t, c0);
            } else {
                zero_row(kk); zero_row(ra);
            }
            b_col(sm + tcs::kBVc, 64, t, c0, kk);
            b_col(sm + tcs::kBdOc, 64, t, c0, ra);
        }
        // Lk V and Mc^T dO need no T: they run while the threads form it (the inverse's
        // scratch is the T tiles' space, which these products do not read); the decay
        // table's row copies have read the plain buffer before the inverse writes it
        bulk_wait_read<0>();
        mma_issue([&](int who) {
            if (who == 0) mma_group(tmem, 128, 64, sbase + tcs::kBVc, tcg::kAtom64, 64, 64);   // Lk V (top)
            else mma_group(tmem, 192, 64, sbase + tcs::kBdOc, tcg::kAtom64, 64, 64);           // Mc^T dO (bottom)
        });
        unit_lower_inverse<kGradThreads>(P1p, P0, reinterpret_cast<float *>(sm + tcs::kBTt));
        if (top) {
#pragma unroll
            for (int i = 0; i < kGW; ++i) x[i] = P0[(c0 + i) * kLD + t];
            b_row(sm + tcs::kBTt, 64, t, c0, x);  // rows t: T[s][t]
        } else {
            plain_row(x, P0, t, c0);
            b_row(sm + tcs::kBTn, 64, t, c0, x);  // rows t: T[t][s]
        }
        ok = mma_stage(bar, phase, p.status, [&](int who) {
            if (who == 0) mma_group(tmem, 0, 384, sbase + tcs::kBTt, tcg::kAtom64, 64, 64);  // W1 = Cm^T T (top)
            else mma_group(tmem, 256, 384, sbase + tcs::kBTn, tcg::kAtom64, 64, 64);         // W2 = Q^T T^T (bottom)
        });
        // T for the gradient pass, one 256-byte bulk copy per row (the stage's barrier and
        // proxy fence published it; nothing writes the plain buffer again)
        if (tid < kC)
            bulk_store(p.Tck + cidx + tid * kN, sbase + tcs::kPlain0 + (uint32_t)(tid * kLD * sizeof(float)),
                       kN * sizeof(float));
        bulk_commit();
    }

    if (ok) {
        // ---- (Lk V)^c, (Mc^T dO)^c; W1, W2 rounded to tf32 in place
        if (top) {
            tmem_ld_row(tl + 128, v);
            b_col(sm + tcs::kBT1, 64, t, c0, v);
            tmem_ld_row(tl + 0, v);
            a_row(tl + 0, v);
        } else {
            tmem_ld_row(tl + 192, v);
            b_col(sm + tcs::kBT1 + 16384, 64, t, c0, v);
            tmem_ld_row(tl + 256, v);
            a_row(tl + 256, v);
        }
        ok = mma_stage(bar, phase, p.status, [&](int who) {
            if (who == 0) {
                mma_group_acc(tmem, 64, 448, sbase + tcs::kBVc, tcg::kAtom64, 64, 64, false, false);    // K^T V
                mma_group_acc(tmem, 64, 0, sbase + tcs::kBT1, tcg::kAtom64, 64, 64, true, true);        // - W1 (Lk V)
                mma_group(tmem, 192, 0, sbase + tcs::kBQc, tcg::kAtom64, 64, 64);                       // W1 Q
            } else {
                mma_group_acc(tmem, 128, 448, sbase + tcs::kBdOc, tcg::kAtom64, 64, 64, false, false);  // R^T dO
                mma_group_acc(tmem, 128, 256, sbase + tcs::kBT1 + 16384, tcg::kAtom64, 64, 64, true,
                              true);                                                                    // - W2 (Mc^T dO)
            }
        });
    }

    if (ok) {
        // ---- out: row i = t of F and A (top), of E (bottom), staged in shared memory (the
        // stage-3 operands are consumed) and written by one 256-byte bulk copy per row
        float *const stage = reinterpret_cast<float *>(sm + tcs::kStage);
        const int i = t;
        if (top) {
            const float sr = __expf(gC[i] - rho[i]);
            tmem_ld_row(tl + 64, v);
#pragma unroll
            for (int j = 0; j < kGW; ++j) v[j] *= sr;
            plain_row_store(stage + 0 * kMat, i, c0, v);
            tmem_ld_row(tl + 192, v);
#pragma unroll
            for (int j = 0; j < kGW; ++j) v[j] = sr * ((c0 + j == i ? 1.f : 0.f) - v[j]) * __expf(rho[c0 + j]);
            plain_row_store(stage + 1 * kMat, i, c0, v);
        } else {
            const float sr = __expf(rho[i]);
            tmem_ld_row(tl + 128, v);
#pragma unroll
            for (int j = 0; j < kGW; ++j) v[j] *= sr;
            plain_row_store(stage + 2 * kMat, i, c0, v);
        }
        fence_proxy_async_smem();
        __syncthreads();
        for (int j = tid; j < 3 * kN; j += kGradThreads) {
            const int gi = j / kN, row = j % kN;
            float *const dst = gi == 0 ? p.Fck : gi == 1 ? p.Ack : p.Eck;
            bulk_store(dst + cidx + row * kN, sbase + tcs::kStage + (uint32_t)((gi * kMat + row * kLD) * sizeof(float)),
                       kN * sizeof(float));
        }
        bulk_commit();
    }
    bulk_wait_read<0>();  // T's and the outputs' row copies have read their tiles (also after a timeout)
    if (tid == 0) {  // the tiles have landed before the shared memory goes away
        mbar_wait_bounded(bar_x, 0, tcg::kMaxPolls);
        mbar_wait_bounded(bar_v, 0, tcg::kMaxPolls);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, tcg::kTmemCols);
}
// ---------------------------------------------------------------------------
// 3. chains over the chunks of one (sequence, head): blockIdx.z = 0 runs the
// states forward (S_{c+1} = A_c S_c + F_c, every boundary stored), 1 runs the
// adjoint backward (Ghat_{c-1} = A_c^T Ghat_c + E_c; Ghat_c stored over E_c).

__global__ void __launch_bounds__(kThreads) bwd_chain_kernel(BwdArgs p) {
    extern __shared__ __align__(16) float sm[];
    float *Am = sm, *Xm = sm + kMat, *Sm = sm + 2 * kMat;
    const int s = blockIdx.x, h = blockIdx.y;
    const bool adjoint = blockIdx.z == 1;
    const int c0 = p.chunk_base[s], nch = p.chunk_base[s + 1] - c0;
    const size_t pair = ((size_t)s * p.H + h) * kStateElems;
    const float *init = adjoint ? (p.dsf ? p.dsf + pair : nullptr) : (p.s0 ? p.s0 + pair : nullptr);
    const float *X = adjoint ? p.Eck : p.Fck;
    load_state(Sm, init);
    __syncthreads();
    if (!adjoint) store_state(p.Sck + ((size_t)(c0 + s) * p.H + h) * kStateElems, Sm);
    // The next step's A and F (or E) are fetched into registers while this step multiplies.
    float4 pa[4], px[4];
    const auto fetch = [&](int step) {
        const int ci = adjoint ? nch - 1 - step : step;
        const size_t cidx = ((size_t)(c0 + ci) * p.H + h) * kStateElems;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = threadIdx.x + q * kThreads, row = e >> 4, c4 = (e & 15) * 4;
            pa[q] = __ldg(reinterpret_cast<const float4 *>(p.Ack + cidx + row * kN + c4));
            px[q] = __ldg(reinterpret_cast<const float4 *>(X + cidx + row * kN + c4));
        }
    };
    if (nch > 0) fetch(0);
    for (int step = 0; step < nch; ++step) {
        const int ci = adjoint ? nch - 1 - step : step;
        const size_t cidx = ((size_t)(c0 + ci) * p.H + h) * kStateElems;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = threadIdx.x + q * kThreads, row = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4 *>(Am + row * kLD + c4) = pa[q];
            *reinterpret_cast<float4 *>(Xm + row * kLD + c4) = px[q];
        }
        __syncthreads();
        if (step + 1 < nch) fetch(step + 1);
        float acc[4][4];
        const int m0 = tile_row(), n0 = tile_col();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 x = *reinterpret_cast<const float4 *>(Xm + (m0 + i) * kLD + n0);
            acc[i][0] = x.x; acc[i][1] = x.y; acc[i][2] = x.z; acc[i][3] = x.w;
        }
        if (adjoint) {
            mm<true, false>(acc, Am, Sm, 0, kC);
            store_state(p.Eck + cidx, Sm);  // the adjoint at this chunk's end (E already read)
        } else {
            mm<false, false>(acc, Am, Sm, 0, kC);
        }
        __syncthreads();
        tile_store(Sm, acc);
        if (!adjoint) {  // the state at this chunk's end, from this thread's own tile (the
                         // next step's barrier publishes the shared copy)
            float *dst = p.Sck + ((size_t)(c0 + s + ci + 1) * p.H + h) * kStateElems;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4 *>(dst + (m0 + i) * kN + n0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
    }
    __syncthreads();  // the last step's shared copy of the state
    if (adjoint && p.ds0) store_state(p.ds0 + pair, Sm);
}

// ---------------------------------------------------------------------------
// 4. per-chunk gradients, on the tensor cores (tcgen05, tf32 operands, fp32
// accumulation in tensor memory).
//
// Every product is one M = 128 MMA whose A operand sits in tensor memory (row m
// in lane m) and whose B operand is a K-major 128-byte-swizzled tile in shared
// memory (D = A B^T).  Two 64-row matrices share one MMA by taking the two
// halves of the lanes: either the same B serves both (stacked rows), or two
// MMAs with different B read the same A columns and each keeps one half.
// Thread (warp w, lane l) owns TMEM lane L = 32 (w mod 4) + l, i.e. row
// t = L mod 64 of the top (L < 64) or bottom matrix, and the 32 columns of half
// w / 4 of every 64-column block.  Transposed operands come from a second MMA
// (C^T = B A^T) or from transposed stores into the B tile, never from moving
// data between lanes.
//
// Stages (each: operands written -> two threads issue their groups -> each commits -> all wait):
//   1  G1 = [Q; Cm] x [Cm; K; R]^T -> Lc, Lk (top), Mc^T (bottom);
//      G2 = K x [R; Q]^T            -> Mk^T, Lk^T (top)
//   2  Y  = [Q | Lk] x [S0'^T | V^c]^T (top);  Y2 = [Cm | Mc^T] x [G'^T | dO^c]^T (bottom)
//   3  U  = T^T Y2 (top), Z = T Y (bottom), from one A holding T^T / T
//   4  dV = [K | Mk^T | -Lk^T] x [G'^T | dO^c | U^c]^T;  P = [V; Z] x [dO; U]^T
//   5  Pt = [U; dO] x [V; Z]^T                           (the transposed P blocks)
//   6  [dK; dC]  = [V | P1 | -P2 ; Z | P3 | -P4] x [G' | R^c | Q^c]^T
//      [dKr; dR] = [U | P2^T | -P4^T ; dO | P1^T | -P3^T] x [S0' | K^c | Cm^T]^T
// then the epilogue scales by the decay factors and forms dr, dk, dkk, da, dw.

__global__ void __launch_bounds__(kGradThreads, 1) bwd_grad_tc_kernel(const __grid_constant__ BwdArgs p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Chunk c;
    if (!locate(p, blockIdx.x, c)) return;
    const int h = blockIdx.y;
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hh = warp >> 2;
    const int L = 32 * quad + lane, t = L & 63, c0 = kGW * hh;
    const bool top = L < 64;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    float *rho = reinterpret_cast<float *>(sm + tcg::kVec), *gC = rho + 64, *carry = gC + 64;  // carry[kGroups][64]
    float *P0 = reinterpret_cast<float *>(sm + tcg::kPlain0);
    const uint32_t bar = sbase + tcg::kBar, bar_st = sbase + tcg::kBar + 16, bar_t = sbase + tcg::kBar + 24,
                   bar_g = sbase + tcg::kBar + 32, bar_x = sbase + tcg::kBar + 40, bar_v = sbase + tcg::kBar + 48,
                   bar_e = sbase + tcg::kBar + 56;
    const size_t cidx = ((size_t)blockIdx.x * p.H + h) * kStateElems;
    const size_t b0 = ((size_t)(blockIdx.x + c.seq) * p.H + h) * kStateElems;
    const size_t b1 = b0 + (size_t)p.H * kStateElems;
    const bool row_valid = t < c.len;
    const size_t roff = ((size_t)(c.tb + (row_valid ? t : 0)) * p.H + h) * kN + c0;  // this thread's token row, half

    if (tid == 0) {
        mbar_init(bar, kIssuers);
        mbar_init(bar_st, 1);
        mbar_init(bar_t, 1);
        mbar_init(bar_g, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_e, 1);
        fence_mbar_init();
        issue_raw_tiles(p, c, h, sbase + tcg::kBG, bar_x);  // B_G's space, written after they are read
        issue_vdo_tiles(p, c, h, sbase + tcg::kVt, sbase + tcg::kPlain1, bar_v, p.x_bf16);
        // the decay table (from the summary pass; unpadded) into the plain buffer, and
        // later into the epilogue's space: phases 0 and 1 of bar_g
        mbar_arrive_expect_tx(bar_g, kStateElems * sizeof(float));
        bulk_load(sbase + tcg::kPlain0, p.Gck + cidx, kStateElems * sizeof(float), bar_g);
        mbar_arrive_expect_tx(bar_st, 3 * kStateElems * sizeof(float));
        bulk_load(sbase + tcg::kSt0, p.Sck + b0, kStateElems * sizeof(float), bar_st);
        bulk_load(sbase + tcg::kSt1, p.Eck + cidx, kStateElems * sizeof(float), bar_st);
        bulk_load(sbase + tcg::kSt2, p.Sck + b1, kStateElems * sizeof(float), bar_st);
    }
    if (warp == 0) tmem_alloc(sbase + tcg::kBar + 8, tcg::kTmemCols);
    // this thread's rows for the scaled operands, from the raw tiles
    float kk[kGW], ra[kGW], rb[kGW];  // top: kk, k; bottom: kk, a, r
    __syncthreads();  // the mbarriers are initialised
    if (!mbar_wait_bounded(bar_x, 0, tcg::kMaxPolls)) report(p.status, kDevTimeout);
    raw_start_rows(kk, ra, rb, sm + tcg::kBG, p.x_bf16, top, row_valid, t, c0);
    const bool got_g = mbar_wait_bounded(bar_g, 0, tcg::kMaxPolls);
    if (!got_g && tid == 0) report(p.status, kDevTimeout);
    if (tid < 64) {
        rho[tid] = P0[31 * kN + tid];
        gC[tid] = P0[63 * kN + tid];
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + tcg::kBar + 8);
    const uint32_t tl = tmem + lane_off + c0;  // this thread's lane, column half
    uint32_t phase = 0;
    bool ok = true;
    float v[kGW], x[kGW];

    // ---- scaled operands: top rows Q, K; bottom rows Cm, R
    {
        float g[kGW], gx[kGW];
        staged_row16(g, P0, t, c0);  // the decay table, unpadded
        if (t > 0) staged_row16(gx, P0, t - 1, c0); else zero_row(gx);
        if (top) {
#pragma unroll
            for (int i = 0; i < kGW; ++i) {
                const float rh = rho[c0 + i];
                v[i] = kk[i] * __expf(gx[i] - rh);     // Q
                x[i] = ra[i] * __expf(rh - g[i]);      // K
            }
            a_row(tl + 0, v);
            a_row(tl + 256, x);
            b_row(sm + tcg::kBG, 256, 64 + t, c0, x);
            b_row(sm + tcg::kBG, 256, 192 + t, c0, v);
            b_col(sm + tcg::kBF1, 64, 128 + t, c0, v);  // Q^c
            b_col(sm + tcg::kBF2, 64, 64 + t, c0, x);   // K^c
        } else {
#pragma unroll
            for (int i = 0; i < kGW; ++i) {
                const float rh = rho[c0 + i];
                v[i] = kk[i] * ra[i] * __expf(rh - g[i]);  // Cm
                x[i] = rb[i] * __expf(g[i] - rh);          // R
            }
            a_row(tl + 0, v);
            b_row(sm + tcg::kBG, 256, t, c0, v);
            b_row(sm + tcg::kBG, 256, 128 + t, c0, x);
            b_col(sm + tcg::kBF1, 64, 64 + t, c0, x);   // R^c
            b_col(sm + tcg::kBF2, 64, 128 + t, c0, v);  // Cm^c
        }
    }
    // fp32 v rows (bottom), in flight during the Gram products (bf16 v and dO come as
    // tiles, the top rows' states by bulk copy)
    if (!top && !p.x_bf16) {
        if (row_valid) load_row(kk, p.v, false, roff);
        else zero_row(kk);
    }
    ok = mma_stage(bar, phase, p.status, [&](int who) {
        if (who == 0) mma_group(tmem, 64, 0, sbase + tcg::kBG, tcg::kAtom256, 192, 64);
        else mma_group(tmem, 320, 256, sbase + tcg::kBG + 128 * 128, tcg::kAtom256, 128, 64);
    });
    // T from the summary pass into the plain buffer (the cumulative decay there has been
    // read), unpadded, in flight during the Gram readout and the B tiles
    bool t_issued = false;
    if (ok && tid == 0) {
        mbar_arrive_expect_tx(bar_t, kStateElems * sizeof(float));
        bulk_load(sbase + tcg::kPlain0, p.Tck + cidx, kStateElems * sizeof(float), bar_t);
        t_issued = true;
    }

    if (ok) {
        // ---- Grams out: A_YY2 = [Q | Lk] (top), [Cm | Mc^T] (bottom); A_F3 = [K | Mk^T | -Lk^T]
        if (top) {  // (L_c, in columns 64.., is not needed here: T comes from the summary pass)
            tmem_ld16x2(tl + 128, tl + 320, x, v);
            mask_row<kStrictLower, false>(x, t, c0);
            a_row_issue(tl + 64, x);
            mask_row<kUpper, false>(v, t, c0);
            a_row_issue(tl + 320, v);
            tmem_ld_row(tl + 384, x);
            mask_row<kStrictUpper, true>(x, t, c0);
            a_row_issue(tl + 384, x);
        } else {
            tmem_ld_row(tl + 192, v);
            mask_row<kUpper, false>(v, t, c0);
            a_row_issue(tl + 64, v);
        }
        tmem_wait_st();
        bool got = true;
        if (top) {  // this row of S0, Ghat and S_C
            got = mbar_wait_bounded(bar_st, 0, tcg::kMaxPolls);
            staged_row16(kk, reinterpret_cast<const float *>(sm + tcg::kSt0), t, c0);
            staged_row16(ra, reinterpret_cast<const float *>(sm + tcg::kSt1), t, c0);
            staged_row16(rb, reinterpret_cast<const float *>(sm + tcg::kSt2), t, c0);
        }
        // B_G no longer read; the staged states read (B_F1 and B_F2 go over them)
        if (!__syncthreads_and(got ? 1 : 0)) {
            if (tid == 0) report(p.status, kDevTimeout);
            ok = false;
        }
    }
    if (ok) {
        // ---- B tiles from the states, V and dO; the carry rowsum(Ghat .* S_C)
        if (top) {
            float part = 0.f;
            const float s0s = __expf(rho[t]), gs = __expf(gC[t] - rho[t]);
#pragma unroll
            for (int i = 0; i < kGW; ++i) {
                part = fmaf(ra[i], rb[i], part);
                kk[i] *= s0s;  // S0'
                ra[i] *= gs;   // G'
            }
            carry[hh * 64 + t] = part;
            b_col(sm + tcg::kBY, 64, t, c0, kk);         // S0'^T
            b_row(sm + tcg::kBF2, 64, t, c0, kk);        // S0'
            b_col(sm + tcg::kBF3, 64, t, c0, ra);        // G'^T
            b_row(sm + tcg::kBF1, 64, t, c0, ra);        // G'
        } else {
            if (!mbar_wait_bounded(bar_v, 0, tcg::kMaxPolls)) report(p.status, kDevTimeout);
            if (row_valid) {  // this row of dO (and of v, bf16)
                if (p.x_bf16) raw_row16(kk, sm + tcg::kVt, true, t, c0);
                raw_row16(ra, sm + tcg::kPlain1, false, t, c0);
            } else {
                zero_row(kk); zero_row(ra);
            }
            b_col(sm + tcg::kBY, 64, 64 + t, c0, kk);    // V^c
            b_col(sm + tcg::kBF3, 64, 64 + t, c0, ra);   // dO^c
        }
        ok = mma_stage(bar, phase, p.status, [&](int who) {
            if (who == 0) mma_group(tmem, 128, 0, sbase + tcg::kBY, tcg::kAtom64, 64, 128);  // Y
            else mma_group(tmem, 192, 0, sbase + tcg::kBF3, tcg::kAtom64, 64, 128);          // Y2
        });
    }

    if (ok) {
        // ---- Y -> Y^c, Y2 -> Y2^c; T rows (cols 0..63) and T^T rows (64..127) in the top lanes
        if (top) {
            tmem_ld_row(tl + 128, v);
            b_col(sm + tcg::kBY, 64, t, c0, v);
            if (!mbar_wait_bounded(bar_t, 0, tcg::kMaxPolls)) report(p.status, kDevTimeout);
            staged_row16(x, P0, t, c0);  // T, unpadded
            a_row(tl + 0, x);
#pragma unroll
            for (int i = 0; i < kGW; ++i) x[i] = P0[(c0 + i) * kN + t];
            a_row(tl + 64, x);
        } else {
            tmem_ld_row(tl + 192, v);
            b_col(sm + tcg::kBY + 16384, 64, t, c0, v);
        }
        ok = mma_stage(bar, phase, p.status, [&](int who) {
            if (who == 0) mma_group(tmem, 128, 0, sbase + tcg::kBY, tcg::kAtom64, 64, 64);  // Z = T Y (top)
            else mma_group(tmem, 192, 64, sbase + tcg::kBY + 16384, tcg::kAtom64, 64, 64);  // U = T^T Y2 (top)
        });
    }

    if (ok) {
        // ---- Z and U out; A_P = [Z; V], A_Pt = [U; dO], B_P = [dO; U], B_Pt = [V; Z], U^c into B_F3
        unsigned char *bp = sm + tcg::kBY, *bpt = sm + tcg::kPlain0;
        if (top) {
            tmem_ld_row(tl + 128, v);  // Z row t
            tmem_ld_row(tl + 192, x);  // U row t
            a_row(tl + 0, v);
            b_row(bpt, 128, 64 + t, c0, v);
            b_col(sm + tcg::kBF3, 64, 128 + t, c0, x);
            b_row(bp, 128, 64 + t, c0, x);
            a_row(tl + 448, x);
        } else {
            a_row(tl + 0, kk);           // V
            b_row(bpt, 128, t, c0, kk);
            b_row(bp, 128, t, c0, ra);   // dO
            a_row(tl + 448, ra);
        }
        ok = mma_stage(bar, phase, p.status, [&](int who) {
            if (who == 0) mma_group(tmem, 192, 256, sbase + tcg::kBF3, tcg::kAtom64, 64, 192);  // dV (top)
            else mma_group(tmem, 64, 0, sbase + tcg::kBY, tcg::kAtom128, 128, 64);              // P
        });
    }

    if (ok) {
        // dV row t into B_F3 (consumed by stage 4); the stage's barrier and proxy fence
        // publish it, and one bulk copy per row writes it out beside the masks below
        if (top) {
            tmem_ld_row(tl + 192, v);  // dV row t
            plain_row_store(reinterpret_cast<float *>(sm + tcg::kDv), t, c0, v);
        }
        ok = mma_stage(bar, phase, p.status, [&](int who) {
            if (who == 0) mma_group(tmem, 320, 448, sbase + tcg::kPlain0, tcg::kAtom128, 128, 64);  // Pt
        });
        if (tid < c.len)
            bulk_store(p.dv + ((size_t)(c.tb + tid) * p.H + h) * kN,
                       sbase + tcg::kDv + (uint32_t)(tid * kLD * sizeof(float)), kN * sizeof(float));
        bulk_commit();
    }

    if (ok) {
        // ---- masks in place: A_F1 = [Z | P3 | -P4 ; V | P1 | -P2] at 0, A_F2 = [U | P2^T | -P4^T ; dO | P1^T | -P3^T] at 256
        tmem_ld16x2(tl + 64, tl + 128, v, x);
        mask_row<kUpper, false>(v, t, c0);
        a_row_issue(tl + 64, v);
        mask_row<kStrictUpper, true>(x, t, c0);
        a_row_issue(tl + 128, x);
        float g3[kGW];
        tmem_ld16x3(tl + 320, tl + 384, tl + 448, v, x, g3);
        if (top) {
            mask_row<kStrictLower, false>(v, t, c0);
            mask_row<kStrictLower, true>(x, t, c0);
        } else {
            mask_row<kLower, false>(v, t, c0);
            mask_row<kLower, true>(x, t, c0);
        }
        a_row_issue(tl + 320, v);
        a_row_issue(tl + 384, x);
        a_row_issue(tl + 256, g3);
        tmem_wait_st();
    }
    bool g2_issued = false;
    if (ok) {
        // the epilogue's rows (top kk, a; bottom r, k: bf16 as tiles into the plain buffers,
        // which B_Pt no longer needs; fp32 per thread) and the decay table again (B_P's space
        // is free), in flight during the last products
        if (!p.x_bf16) {
            if (row_valid) {
                load_row(kk, top ? p.kk : p.r, false, roff);
                load_row(ra, top ? p.a : p.k, false, roff);
            } else {
                zero_row(kk); zero_row(ra);
            }
        }
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_g, kStateElems * sizeof(float));
            bulk_load(sbase + 0, p.Gck + cidx, kStateElems * sizeof(float), bar_g);
            g2_issued = true;
            if (p.x_bf16) issue_raw_tiles(p, c, h, sbase + tcg::kPlain0, bar_e);
        }
        bulk_wait_read<0>();  // dV's tile is read before the epilogue writes over it
        ok = mma_stage(bar, phase, p.status, [&](int who) {
            if (who == 0) mma_group(tmem, 192, 0, sbase + tcg::kBF1, tcg::kAtom64, 64, 192);  // [dC; dK]
            else mma_group(tmem, 448, 256, sbase + tcg::kBF2, tcg::kAtom64, 64, 192);         // [dKr; dR]
        });
    }

    if (ok) {
        // ---- epilogue: top rows hold dC, dKr; bottom rows dK, dR.  Each half writes its
        // part of W = r dr - k dk - c dC + kk dKr; the reverse cumulative sum adds them.
        const float *Gm = reinterpret_cast<const float *>(sm + 0);  // the decay table, unpadded
        float *PW = reinterpret_cast<float *>(sm + 17408);  // top part, then the cumulative sum
        float *PB = reinterpret_cast<float *>(sm + 34816);  // bottom part
        float *const stage = reinterpret_cast<float *>(sm + tcg::kStage);
        if (!mbar_wait_bounded(bar_g, 1, tcg::kMaxPolls)) report(p.status, kDevTimeout);
        if (p.x_bf16) {  // this row of kk, a (top) or r, k (bottom) from the tiles
            if (!mbar_wait_bounded(bar_e, 0, tcg::kMaxPolls)) report(p.status, kDevTimeout);
            if (row_valid) {
                const unsigned char *tl0 = sm + tcg::kPlain0;  // kk, k, a, r, 8 KB apart
                raw_row16(kk, tl0 + (top ? 0 : 3) * 8192, true, t, c0);
                raw_row16(ra, tl0 + (top ? 2 : 1) * 8192, true, t, c0);
            } else {
                zero_row(kk); zero_row(ra);
            }
        }
        float g[kGW], acc1[kGW], acc2[kGW];
        staged_row16(g, Gm, t, c0);
        tmem_ld_row(tl + 192, acc1);  // top dC, bottom dK
        tmem_ld_row(tl + 448, acc2);  // top dKr, bottom dR
        float Y[kGW];
        if (top) {
            float gx[kGW];
            if (t > 0) staged_row16(gx, Gm, t - 1, c0); else zero_row(gx);
#pragma unroll
            for (int i = 0; i < kGW; ++i) {
                const float rh = rho[c0 + i];
                const float dC = -acc1[i] * __expf(rh - g[i]);
                const float dKr = -acc2[i] * __expf(gx[i] - rh);
                Y[i] = kk[i] * dKr;
                x[i] = Y[i] - kk[i] * ra[i] * dC;  // - c dC + kk dKr
                acc1[i] = kk[i] * dC;              // da
                acc2[i] = dKr + ra[i] * dC;        // dkk
            }
            plain_row_store(PW, t, c0, x);
            plain_row_store(stage + 0 * kMat, t, c0, acc1);
            plain_row_store(stage + 1 * kMat, t, c0, acc2);
        } else {
#pragma unroll
            for (int i = 0; i < kGW; ++i) {
                const float rh = rho[c0 + i];
                const float dK = acc1[i] * __expf(rh - g[i]);
                const float dR = acc2[i] * __expf(g[i] - rh);
                x[i] = kk[i] * dR - ra[i] * dK;  // r dr - k dk
                acc1[i] = dK;
                acc2[i] = dR;
            }
            plain_row_store(PB, t, c0, x);
            plain_row_store(stage + 2 * kMat, t, c0, acc1);
            plain_row_store(stage + 3 * kMat, t, c0, acc2);
        }
        __syncthreads();
        {
            // reverse inclusive cumulative sum over tokens per channel, plus the carry
            float *scratch = reinterpret_cast<float *>(sm + 52224);
            constexpr int kSeg = kGradThreads / 64, kRows = 64 / kSeg;  // row segments of the sum
            const int ch = tid & 63, qt = tid >> 6;
            float run = 0.f;
            float part[kRows];
#pragma unroll
            for (int u = kRows - 1; u >= 0; --u) {
                run += PW[(qt * kRows + u) * kLD + ch] + PB[(qt * kRows + u) * kLD + ch];
                part[u] = run;
            }
            scratch[qt * kLD + ch] = run;
            __syncthreads();
            float base = 0.f;
#pragma unroll
            for (int q = 0; q < kGroups; ++q) base += carry[q * 64 + ch];
            for (int q = qt + 1; q < kSeg; ++q) base += scratch[q * kLD + ch];
#pragma unroll
            for (int u = 0; u < kRows; ++u) PW[(qt * kRows + u) * kLD + ch] = part[u] + base;
            __syncthreads();
        }
        if (top) {
            plain_row(v, PW, t, c0);
#pragma unroll
            for (int i = 0; i < kGW; ++i) v[i] -= Y[i];
            plain_row_store(stage + 4 * kMat, t, c0, v);
        }
        // every valid row of the five tiles leaves by one 256-byte bulk copy (a warp's own
        // stores would touch 32 rows each)
        fence_proxy_async_smem();
        __syncthreads();
        for (int i = tid; i < 5 * kC; i += kGradThreads) {
            const int gi = i / kC, row = i % kC;
            float *const dst = gi == 0 ? p.da : gi == 1 ? p.dkk : gi == 2 ? p.dk : gi == 3 ? p.dr : p.dw;
            if (row < c.len)
                bulk_store(dst + ((size_t)(c.tb + row) * p.H + h) * kN,
                           sbase + tcg::kStage + (uint32_t)((gi * kMat + row * kLD) * sizeof(float)), kN * sizeof(float));
        }
        bulk_commit();
    }
    bulk_wait_read<0>();  // every row copy has read its tile (also after a timeout)
    if (tid == 0) {  // every bulk copy and TMA tile has landed before the shared memory goes away
        mbar_wait_bounded(bar_st, 0, tcg::kMaxPolls);
        if (t_issued) mbar_wait_bounded(bar_t, 0, tcg::kMaxPolls);
        mbar_wait_bounded(bar_x, 0, tcg::kMaxPolls);
        mbar_wait_bounded(bar_g, g2_issued ? 1 : 0, tcg::kMaxPolls);
        mbar_wait_bounded(bar_v, 0, tcg::kMaxPolls);
        if (g2_issued && p.x_bf16) mbar_wait_bounded(bar_e, 0, tcg::kMaxPolls);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, tcg::kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
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

// 2-D map over a packed [T_total, H*64] input: 64-row boxes of 128-byte rows (64 bf16 or
// 32 fp32 channels) in the 128-byte swizzle layout.
bool make_tile_map(CUtensorMap *map, const void *base, bool bf16, int T_total, int H) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * 64, static_cast<cuuint64_t>(T_total)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 64 * esz};
    cuuint32_t box[2] = {bf16 ? 64u : 32u, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

// Upper bound on the chunks of any packing of T_total tokens into num_seqs sequences.
long long prefill_backward_max_chunks(int num_seqs, int T_total) { return (long long)T_total / kC + num_seqs; }

size_t prefill_backward_workspace_bytes(int num_seqs, int T_total, int H) {
    const long long nc = prefill_backward_max_chunks(num_seqs, T_total);
    const size_t table = ((size_t)(num_seqs + 1) * sizeof(int32_t) + 255) & ~(size_t)255;
    const size_t mat = kStateElems * sizeof(float);
    return table + (size_t)(6 * nc + num_seqs) * H * mat;
}

cudaError_t launch_prefill_backward(const BackwardArgs &b, void *workspace, cudaStream_t stream) {
    static int attr_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_dev != dev) {
        e = cudaFuncSetAttribute(bwd_summary_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcs::kAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bwd_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcg::kAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kChainSmem);
        if (e != cudaSuccess) return e;
        attr_dev = dev;
    }
    const long long nc = prefill_backward_max_chunks(b.num_seqs, b.T_total);
    const size_t table = ((size_t)(b.num_seqs + 1) * sizeof(int32_t) + 255) & ~(size_t)255;
    const size_t plane = (size_t)b.H * kStateElems;
    char *ws = static_cast<char *>(workspace);
    BwdArgs p;
    p.num_seqs = b.num_seqs;
    p.H = b.H;
    p.cu = b.cu_seqlens;
    p.x_bf16 = b.x_dtype == WKV7_BF16;
    p.r = b.r; p.k = b.k; p.v = b.v; p.kk = b.kk; p.a = b.a; p.w = b.w;
    p.s0 = b.initial_state;
    p.d_o = b.d_o;
    p.dsf = b.d_final_state;
    p.dr = b.dr; p.dw = b.dw; p.dk = b.dk; p.dv = b.dv; p.dkk = b.dkk; p.da = b.da;
    p.ds0 = b.d_initial_state;
    p.status = b.status;
    p.chunk_base = reinterpret_cast<int32_t *>(ws);
    p.Sck = reinterpret_cast<float *>(ws + table);
    p.Ack = p.Sck + (size_t)(nc + b.num_seqs) * plane;
    p.Fck = p.Ack + (size_t)nc * plane;
    p.Eck = p.Fck + (size_t)nc * plane;
    p.Tck = p.Eck + (size_t)nc * plane;
    p.Gck = p.Tck + (size_t)nc * plane;

    if (nc > 0 && (!make_tile_map(&p.mkk, b.kk, p.x_bf16, b.T_total, b.H) ||
                   !make_tile_map(&p.mk, b.k, p.x_bf16, b.T_total, b.H) ||
                   !make_tile_map(&p.ma, b.a, p.x_bf16, b.T_total, b.H) ||
                   !make_tile_map(&p.mr, b.r, p.x_bf16, b.T_total, b.H) ||
                   !make_tile_map(&p.mv, b.v, p.x_bf16, b.T_total, b.H) ||
                   !make_tile_map(&p.mdo, b.d_o, false, b.T_total, b.H)))
        return cudaErrorInvalidValue;
    bwd_chunk_table_kernel<<<1, 1024, 0, stream>>>(b.cu_seqlens, b.num_seqs, b.T_total, p.chunk_base, b.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (nc > 0) {
        const dim3 grid((unsigned)nc, (unsigned)b.H);
        bwd_summary_tc_kernel<<<grid, kGradThreads, tcs::kAlloc, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    bwd_chain_kernel<<<dim3((unsigned)b.num_seqs, (unsigned)b.H, 2), kThreads, kChainSmem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (nc > 0) {
        const dim3 grid((unsigned)nc, (unsigned)b.H);
        bwd_grad_tc_kernel<<<grid, kGradThreads, tcg::kAlloc, stream>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace wkv7
