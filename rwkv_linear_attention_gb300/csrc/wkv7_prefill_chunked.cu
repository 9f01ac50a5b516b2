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
// In block form, with W = Qa S0 + L_k V (= T^{-1} Z, which needs no inverse):
//
//   [ O                  ]   [ Ra | M_k  ]   [ S0 ]   [ M_c  ]
//   [ S_C - e^{g_C} * S0 ] = [ 0  | Kb^T ] . [ V  ] - [ Cb^T ] . T W
//
// Every row i of the lower half carries the factor e^{g_C - g_ref}[i]
// (Cb^T = diag(e^{g_C - g_ref}) C^T, likewise Kb^T); the kernel keeps the lower
// half without it and applies it to the state rows of the product.  Every S0
// column i carries the factor e^{g_ref}[i] (Ra = R diag(e^{g_ref}),
// Qa = Q diag(e^{g_ref}), with R and Q the Gram operands below); the kernel
// keeps those columns without it and scales the rows of the state operand
// instead, S0' = diag(e^{g_ref}) S0.  Per chunk these tf32 MMAs run, all with
// M = 128, fp32 accumulators in tensor memory and the A operand read from
// tensor memory:
//   G = [R ; Q] [C ; K]^T                (the four Gram blocks; 128x128x64)
//   W = [R | M_k ; Q | L_k] [S0' ; V]    (rows 64..127 are W, rows 0..63 are not used,
//                                         their M_k unmasked; 128x64x128, needs no T)
//   X = [M_c ; C^T] T                    (three small products, see phase 4)
//   D = [R | M_k ; 0 | K^T] [S0' ; V] - X W   (128x64x128, then 128x64x64)
// so after the T halves only X and the last K = 64 product remain on the
// critical path, and no intermediate carries the e^{64|w|} of the chunk's
// removal block C^T T Q (which the transition contains but no product forms).
// C^T and K^T (the lower lanes of A_X and of the base) are copied from the Gram
// B operand [C ; K] in shared memory into tensor memory by threads, and R (the
// base's upper left block) from the Gram A operand.
// The SIMT work (cumulative decay, exponentials, masks, the blocked 64x64
// unit-lower-triangular inverse, operand staging) is software-pipelined with
// the MMAs: the next chunk's decay and Gram operands are built while this
// chunk's X and D products run, and the next chunk's Gram product runs
// while this chunk's outputs are written.  A dedicated warp issues every MMA and
// every TMA copy (input tiles a chunk ahead, output stores), so no worker
// thread stalls on an issue queue.  One CTA (512 threads) owns one
// (sequence, head) pair and walks its chunks in order; the fp32 state lives
// in registers between chunks.  Inputs arrive by TMA as 2-D tiles of
// 64 tokens x 64 channels of the packed [T, H, 64] arrays (bf16 tiles in the
// 128-byte swizzled layout, so both row- and column-wise reads are free of
// bank conflicts); a chunk's tiles are requested as soon as the previous
// chunk's are consumed, a full chunk before they are needed.
//
// Inputs r, k, v, kk, a are bf16, or fp32 (then read from global memory after
// an L2 prefetch, see kF32In); w is fp32.
//
// Precision: inputs are used exactly; operands staged by threads are rounded
// to tf32 (to nearest); operands that one MMA hands to the next stay in
// tensor memory (the hardware reads them at tf32 precision); accumulation is
// fp32 and the state carried between chunks is fp32.  The decay factors of
// the Gram operands are taken relative to the chunk's 32nd token, so for
// w >= -1 every factor lies within e^{+-32} and every product of two within
// e^{+-64} (finite in fp32); phase 1 reports a w below -1.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <numeric>
#include <vector>

#include "sm103_ptx.cuh"
#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk length
constexpr int kThreads = 512;   // worker warps w < 16: TMEM lane quarter w % 4, column group w / 4
constexpr int kBlock = kThreads + 32;  // + one warp that issues every MMA and TMA copy
constexpr uint32_t kMaxPolls = 1u << 24;

// TMEM columns.  The chunk's outputs and state increment are
//   D = base [S0' ; V] - X W,   base = [R | M_k ; 0 | K^T],  X = [M_c ; Cb^T] T,
//   W = [Q | L_k] [S0' ; V]  (= Q S0' + L_k V, rows 64..127 of an M = 128 product),
// so W needs no T and runs while the T halves are formed; after them only X and
// one K = 64 product remain on the tensor core.  W is written over G's first 64
// columns once they are read, with L_k masked in place beside it as its A operand.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0;     // G; then W in its columns 0..63 (A operand [Q | L_k]: A_G, G 64..127)
constexpr uint32_t kColX = 128;   // X = [Mt ; Ct]
constexpr uint32_t kColAX = 192;  // A_X = [M_c ; C^T], the A operand of X (64 columns)
constexpr uint32_t kColAC = 256;  // the base [R | M_k ; 0 | K^T] (128 columns: the S0 block, then the V block)
constexpr uint32_t kColAG = 384;  // A operand of G = [R ; Q] (for the next chunk)
constexpr uint32_t kColD = 448;   // D = [O ; S_C - e^{g_C} S0]
static_assert(kColX == kColG + 128 && kColAX == kColX + 64 && kColAC == kColAX + 64 && kColAG == kColAC + 128 &&
                  kColD == kColAG + 64 && kColD + 64 <= kTmemCols,
              "tensor-memory regions must tile the allocation without overlap");

constexpr int kLd = 68;  // padded row stride (floats) of the fp32 L_c^T scratch

// Shared memory map (bytes from a 1024-aligned base)
constexpr int kTile = 64 * 64 * 2;  // one bf16 raw tile
constexpr int SM_R = 0, SM_K = SM_R + kTile, SM_KK = SM_K + kTile, SM_A = SM_KK + kTile, SM_V = SM_A + kTile;
constexpr int SM_W = SM_V + kTile;         // fp32 w tile -> E = e^{g - g_ref} (swizzled)
constexpr int SM_BG = SM_W + 16384;        // B operand of G: [C ; K]  (128 x K64)
constexpr int SM_BY = SM_BG + 32768;       // B operand of the last product: W^T (64 x K64; 32 KB reserved)
constexpr int SM_BX = SM_BY + 32768;       // B operand of X: T^T (64 x K64)
constexpr int SM_BC = SM_BX + 16384;       // B operand of D: [S0'^T | V^T] (64 x K128)
constexpr int SM_LC = SM_BC + 32768;       // fp32 L_c^T [64][kLd]
constexpr int SM_TS = SM_LC + 64 * kLd * 4;  // output staging for the TMA stores
constexpr int SM_XS = SM_TS + 64 * kLd * 4;  // fp32 2 x 16 x 16 scratch (T_11 of each half)
constexpr int SM_TOT = SM_XS + 4096;       // 16 x 64 cumsum partials
constexpr int SM_GREF = SM_TOT + 4096;     // 64: g_ref
constexpr int SM_EREF = SM_GREF + 256;     // 2 x 64: e^{g_ref} (double-buffered across chunks)
constexpr int SM_E63 = SM_EREF + 512;      // 2 x 64: e^{g_C - g_ref} (double-buffered across chunks)
constexpr int SM_GC = SM_E63 + 512;        // 2 x 64: e^{g_C} (double-buffered across chunks)
constexpr int SM_BAR = SM_GC + 512;        // 7 mbarriers
constexpr int SM_SLOT = SM_BAR + 128;
static_assert(7 * 8 <= SM_SLOT - SM_BAR, "mbarriers exceed their space");
constexpr int kSmemBytes = SM_SLOT + 64;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory layout too large");
static_assert(SM_BG % 1024 == 0 && SM_BY % 1024 == 0 && SM_BX % 1024 == 0 && SM_BC % 1024 == 0,
              "operand tiles must be 1024-byte aligned");
constexpr uint32_t kTmaBytes = 5 * kTile + 16384;

// An fp32 value as a tf32 MMA operand, rounded to nearest (ties away from zero):
// the tensor core reads the top 19 bits of each 32-bit operand and ignores the low
// 13, so adding half a tf32 ulp (bit 12) to the bit pattern makes that truncation
// round.  Used only for words the tensor core consumes.
__device__ __forceinline__ uint32_t to_tf32(float x) { return __float_as_uint(x) + 0x1000u; }
__device__ __forceinline__ void st_tf32x4(unsigned char *p, float a, float b, float c, float d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(to_tf32(a), to_tf32(b), to_tf32(c), to_tf32(d));
}
// Reciprocal of a decay factor (the hardware approximation, rcp.approx.ftz, ~1 ulp);
// it only feeds tf32 operands, whose rounding dominates.  Factors lie in e^{+-80}.
__device__ __forceinline__ float rcp(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float bf2f(uint32_t lo16) { return __uint_as_float(lo16 << 16); }

// bf16 raw tile [64 tokens][64 channels] in the TMA 128-byte swizzle layout.
__device__ __forceinline__ uint32_t raw_off(int t, int i) {
    return t * 128 + ((((i >> 3) ^ (t & 7)) << 4) | ((i & 7) << 1));
}
// channels i, i+1 (i even)
__device__ __forceinline__ float2 raw2(const unsigned char *tile, int t, int i) {
    const uint32_t u = *reinterpret_cast<const uint32_t *>(tile + raw_off(t, i));
    return make_float2(bf2f(u & 0xffffu), __uint_as_float(u & 0xffff0000u));
}
// four consecutive channels i .. i+3 (i % 4 == 0)
__device__ __forceinline__ float4 raw4(const unsigned char *tile, int t, int i) {
    const uint2 u = *reinterpret_cast<const uint2 *>(tile + raw_off(t, i));
    return make_float4(bf2f(u.x & 0xffffu), __uint_as_float(u.x & 0xffff0000u), bf2f(u.y & 0xffffu),
                       __uint_as_float(u.y & 0xffff0000u));
}
// eight consecutive channels i .. i+7 (i % 8 == 0)
__device__ __forceinline__ void raw8(const unsigned char *tile, int t, int i, float *f) {
    const uint4 u = *reinterpret_cast<const uint4 *>(tile + raw_off(t, i));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = bf2f(w[j] & 0xffffu);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
}
// E table [64][64] fp32 with 16-byte chunks XOR-swizzled by (t mod 8).
__device__ __forceinline__ int eidx(int t, int i) { return t * 64 + ((((i >> 2) ^ (t & 7)) << 2) | (i & 3)); }

struct TensorMaps {
    CUtensorMap r, k, v, kk, a, w;
    CUtensorMap o;     // output: fp32 as 64 x 32 boxes, bf16 as 64 x 64 boxes, 128-byte swizzle (stores)
    CUtensorMap ohat;  // fp32 [rows, 64] carry-in readout of transfer items, same boxes
};

// ---- Tail split.  A CTA runs one work item.  Items 0 .. main_items-1 are whole
// (sequence, head) pairs in schedule order (blockIdx = rank * H + h).  The pairs
// that would run alone in a last, mostly idle wave of CTAs are instead cut into
// k chunk-aligned segments, each running concurrently on its own SM.  The
// recurrence is linear in the state: over a segment, S_end = P S_in + S_part with
// P the product of the per-token transitions diag(e^w) - (kk*a) kk^T, and
// o_t = o_part_t + S_in^T (P_t^T r_t).  So for segment j >= 1 of a split pair
// two items run, one from S = 0 (o_part into o, S_part into a slot) and one from
// S = I with v = 0 (P_t^T r_t into a scratch row, P into a slot); segment 0
// runs from the true initial state.  Two small kernels then chain the true
// boundary states (S_in(j+1) = P(j) S_in(j) + S_part(j)) and add S_in(j)^T
// P_t^T r_t to the outputs of segment j.
enum : int16_t { kItemWhole = 0, kItemPart = 1, kItemTransfer = 2 };
struct SplitItem {
    int32_t pair;       // b * H + h
    int16_t c0, c1;     // chunk range [c0, c1) of the pair
    int16_t kind;       // kItemWhole (segment 0 too), kItemPart, kItemTransfer
    int16_t slot;       // state slot for the final state (-1: the caller's final_state)
    int32_t ohat_row;   // first scratch row of a transfer item's readout, or (bf16 output)
                        // of a part item's fp32 outputs
};
constexpr int kMaxSplitItems = 512;
constexpr int kMaxSplitPairs = 80;
constexpr int kMaxSegs = 16;
struct SplitPlan {
    int main_items;
    int n_items;
    float *slots;   // kMaxSplitItems x 4096 fp32 states
    float *ohat;    // scratch rows x 64 fp32
    SplitItem item[kMaxSplitItems];
};
struct FixSeg {
    int16_t c0, c1;
    int16_t slot_part, slot_transfer;  // slot_part of segment 0: its (true) final state
    int32_t ohat_row;                  // the transfer item's readout rows
    int32_t opart_row;                 // with a bf16 output: the part item's fp32 output rows
};
struct FixPair {
    int32_t b, h, nseg;
    FixSeg seg[kMaxSegs];
};
struct FixPlan {
    int n_pairs;
    int n_blocks;  // output-fix blocks per pair: the most chunks after a first segment
    float *slots;
    float *ohat;
    FixPair pair[kMaxSplitPairs];
};

// Barriers among the 512 worker threads (the MMA warp never joins them).
__device__ __forceinline__ void wsync() { named_sync<1, kThreads>(); }

// All workers wait on an mbarrier phase; the outcome is uniform, so either
// every worker continues or every worker leaves together.
__device__ __forceinline__ bool wait_uniform(uint32_t bar, uint32_t parity, unsigned *status) {
    const bool ok = mbar_wait_bounded(bar, parity, kMaxPolls);
    const int any_fail = named_sync_or<1, kThreads>(ok ? 0 : 1);
    if (any_fail && threadIdx.x == 0) report(status, kDevTimeout);
    return any_fail == 0;
}

// Shared-memory operand writes and tensor-memory stores by all workers ->
// visible to the tensor core and to every worker after this barrier.
__device__ __forceinline__ void sync_for_mma() {
    fence_proxy_async_smem();
    tc_fence_before_sync();
    wsync();
    tc_fence_after_sync();
}

// Operands for the next MMA step are in place: publish them and tell the MMA warp.
__device__ __forceinline__ void handoff(uint32_t rdy) {
    sync_for_mma();
    if (threadIdx.x == 0) mbar_arrive(rdy);
}

// kF32In: r, k, v, kk, a are fp32 (contracted at tf32 like the rest).  Their tiles are twice
// the size of bf16 tiles and do not fit beside the operand buffers, so only w is staged by TMA;
// the other five are prefetched into L2 when w is requested and read from global memory where
// the bf16 form reads its swizzled tiles.
template <bool kF32In>
__global__ void __launch_bounds__(kBlock, 1)
wkv7_prefill_chunked_kernel(PrefillArgs p, const __grid_constant__ TensorMaps maps,
                            const __grid_constant__ SplitPlan plan) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q = warp & 3, cg = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    const int m = 32 * q + lane;  // TMEM lane (row) this thread reads and writes

    const int H = p.H;
    int b, h, c_begin = 0, c_end = -1, kind = kItemWhole, slot = -1, ohat_row = 0;
    if (static_cast<int>(blockIdx.x) < plan.main_items) {
        const int rank = static_cast<int>(blockIdx.x) / H;
        h = static_cast<int>(blockIdx.x) % H;
        b = p.order ? p.order[rank] : rank;
    } else {
        const SplitItem &it = plan.item[blockIdx.x - plan.main_items];
        b = it.pair / H;
        h = it.pair % H;
        c_begin = it.c0;
        c_end = it.c1;
        kind = it.kind;
        slot = it.slot;
        ohat_row = it.ohat_row;
    }
    if (b < 0 || b >= p.num_seqs) {
        if (tid == 0) report(p.status, kDevBounds);
        return;
    }
    int bos, eos;
    seq_bounds(p, b, bos, eos);
    if (bos < 0 || eos < bos || eos > p.T_total || (p.lens && eos - bos > p.row_stride)) {
        if (tid == 0) report(p.status, kDevBadSeqlens);
        return;
    }
    const int len = eos - bos;
    if (c_end < 0) c_end = (len + kC - 1) / kC;
    if (c_begin < 0 || c_end < c_begin || (c_end > c_begin && (c_end - 1) * kC >= len)) {
        if (tid == 0) report(p.status, kDevBadSeqlens);  // the schedule disagrees with the device lengths
        return;
    }
    const int nchunks = c_end - c_begin;  // chunks of this item; loop indices below are relative to c_begin
    const long long tok_stride = static_cast<long long>(H) * 64;
    // outputs that go to fp32 scratch rows: a transfer item's readout, and a part item's
    // partial outputs when o is bf16 (the correction is added before the one rounding)
    const bool to_scratch = kind == kItemTransfer || (kind == kItemPart && p.o_dtype == WKV7_BF16);
    const bool bf16_out = p.o_dtype == WKV7_BF16 && !to_scratch;

    // State: rows i = m - 64 (lanes 64..127), columns 16*cg .. 16*cg+15.
    const bool state_thread = q >= 2;
    const int si = m - 64;
    float s[16];
    const long long sslot = (static_cast<long long>(b) * H + h) * 4096;
    if (state_thread) {
        if (kind == kItemTransfer) {  // S = I
#pragma unroll
            for (int j = 0; j < 16; ++j) s[j] = (16 * cg + j == si) ? 1.f : 0.f;
        } else if (kind == kItemWhole && p.initial_state) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 x = load_state4(p.initial_state, p.state_dtype, sslot + si * 64 + 16 * cg + 4 * j);
                s[4 * j] = x.x; s[4 * j + 1] = x.y; s[4 * j + 2] = x.z; s[4 * j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) s[j] = 0.f;
        }
    }
    if (nchunks == 0) {
        if (state_thread && p.final_state) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                store_state4(p.final_state, p.state_dtype, sslot + si * 64 + 16 * cg + 4 * j,
                             make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]));
        }
        return;
    }

    unsigned char *rr = sm + SM_R, *rk = sm + SM_K, *rkk = sm + SM_KK, *ra = sm + SM_A, *rv = sm + SM_V;
    float *E = reinterpret_cast<float *>(sm + SM_W);
    float *TOT = reinterpret_cast<float *>(sm + SM_TOT);
    float *GREF = reinterpret_cast<float *>(sm + SM_GREF);
    float *EREF = reinterpret_cast<float *>(sm + SM_EREF);
    float *E63 = reinterpret_cast<float *>(sm + SM_E63);
    float *GC = reinterpret_cast<float *>(sm + SM_GC);
    // Product-complete barriers (tensor-core commits) and one operands-ready barrier per
    // handoff from the workers to the MMA warp.  Each handoff barrier completes once per
    // chunk and the workers cannot reach the same handoff of the next chunk before the MMA
    // warp has consumed this one (they first wait on a product it issues after it), so a
    // waiter never misses a phase.
    const uint32_t bar_tma = sbase + SM_BAR, bar_g = bar_tma + 8, bar_d = bar_tma + 16, bar_i = bar_tma + 24;
    const uint32_t rdy_x = bar_tma + 32, rdy_g = bar_tma + 40, rdy_t = bar_tma + 48;
    const uint32_t rdy_w = bar_tma + 56, bar_w = bar_tma + 64;  // W's operands ready; W complete
    const uint32_t rdy_b = bar_tma + 72;                        // the base [R | M_k ; 0 | K^T] ready

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_g, 1);
        mbar_init(bar_d, 1);
        mbar_init(bar_i, 1);
        mbar_init(rdy_x, 1);
        mbar_init(rdy_g, 1);
        mbar_init(rdy_t, 1);
        mbar_init(rdy_w, 1);
        mbar_init(bar_w, 1);
        mbar_init(rdy_b, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(sbase + SM_SLOT, kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + SM_SLOT);

    auto issue_tma = [&](int chunk) {
        const int y = bos + (c_begin + chunk) * kC, x = h * 64;
        if constexpr (kF32In) {
            mbar_arrive_expect_tx(bar_tma, 16384u);
            tma_prefetch_2d(&maps.r, x, y);
            tma_prefetch_2d(&maps.k, x, y);
            tma_prefetch_2d(&maps.kk, x, y);
            tma_prefetch_2d(&maps.a, x, y);
            tma_prefetch_2d(&maps.v, x, y);
        } else {
            mbar_arrive_expect_tx(bar_tma, kTmaBytes);
            tma_load_2d(sbase + SM_R, &maps.r, x, y, bar_tma);
            tma_load_2d(sbase + SM_K, &maps.k, x, y, bar_tma);
            tma_load_2d(sbase + SM_KK, &maps.kk, x, y, bar_tma);
            tma_load_2d(sbase + SM_A, &maps.a, x, y, bar_tma);
            tma_load_2d(sbase + SM_V, &maps.v, x, y, bar_tma);
        }
        tma_load_2d(sbase + SM_W, &maps.w, x, y, bar_tma);
    };
    // Channels i .. of row t of chunk `chunk` of an input: from its staged bf16 tile, or (fp32
    // inputs) from global memory.
    auto xrow = [&](const void *x, int chunk, int t) {
        return static_cast<const float *>(x) + (static_cast<long long>(bos + (c_begin + chunk) * kC + t) * H + h) * 64;
    };
    auto in2 = [&](const unsigned char *tile, const void *x, int chunk, int t, int i) -> float2 {
        if constexpr (kF32In) return __ldg(reinterpret_cast<const float2 *>(xrow(x, chunk, t) + i));
        else return raw2(tile, t, i);
    };
    auto in4 = [&](const unsigned char *tile, const void *x, int chunk, int t, int i) -> float4 {
        if constexpr (kF32In) return __ldg(reinterpret_cast<const float4 *>(xrow(x, chunk, t) + i));
        else return raw4(tile, t, i);
    };
    auto in8 = [&](const unsigned char *tile, const void *x, int chunk, int t, int i, float *f) {
        if constexpr (kF32In) {
            const float4 *src = reinterpret_cast<const float4 *>(xrow(x, chunk, t) + i);
            const float4 u0 = __ldg(src), u1 = __ldg(src + 1);
            f[0] = u0.x; f[1] = u0.y; f[2] = u0.z; f[3] = u0.w;
            f[4] = u1.x; f[5] = u1.y; f[6] = u1.z; f[7] = u1.w;
        } else {
            raw8(tile, t, i, f);
        }
    };
    auto chunk_len = [&](int chunk) { return min(kC, eos - (bos + (c_begin + chunk) * kC)); };

    // ---- phase 1: masked cumulative log-decay g; E = e^{g - g_ref} (g_ref = g[31]) in place.
    // Thread: channels 2cp, 2cp+1 of rows 4 seg .. 4 seg + 3 (16 row segments; their totals
    // are scanned through TOT).
    auto phase1 = [&](int lc, int gbuf) {
        const int ch = 2 * (tid & 31), seg = tid >> 5;
        float2 g[4];
        float2 acc = make_float2(0.f, 0.f);
        float wmin = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = 4 * seg + u;
            if (t < lc) {  // the w tile, row-major as loaded
                const float2 wv = *reinterpret_cast<const float2 *>(E + t * 64 + ch);
                acc.x += wv.x;
                acc.y += wv.y;
                wmin = fminf(wmin, fminf(wv.x, wv.y));
            }
            g[u] = acc;
        }
        if (wmin < kMinLogDecay) report(p.status, kDevDomain);  // outside the domain: reported, not trapped
        *reinterpret_cast<float2 *>(TOT + seg * 64 + ch) = acc;
        wsync();
        float2 pre = make_float2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 15; ++u) {  // unrolled, so that the loads issue back to back
            if (u < seg) {
                const float2 tv = *reinterpret_cast<const float2 *>(TOT + u * 64 + ch);
                pre.x += tv.x;
                pre.y += tv.y;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            g[u].x += pre.x;
            g[u].y += pre.y;
        }
        if (seg == 7) *reinterpret_cast<float2 *>(GREF + ch) = g[3];  // row 31
        wsync();
        const float2 gr = *reinterpret_cast<const float2 *>(GREF + ch);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = 4 * seg + u;
            *reinterpret_cast<float2 *>(E + eidx(t, ch)) = make_float2(__expf(g[u].x - gr.x), __expf(g[u].y - gr.y));
        }
        if (seg == 0) *reinterpret_cast<float2 *>(EREF + gbuf * 64 + ch) = make_float2(__expf(gr.x), __expf(gr.y));
        if (seg == 15) {  // row 63
            *reinterpret_cast<float2 *>(E63 + gbuf * 64 + ch) = make_float2(__expf(g[3].x - gr.x), __expf(g[3].y - gr.y));
            *reinterpret_cast<float2 *>(GC + gbuf * 64 + ch) = make_float2(__expf(g[3].x), __expf(g[3].y));
        }
    };

    // ---- phase 2: A_G = [R ; Q] into TMEM; the Gram B operand B_G = [C ; K] (rows s, 64 + s),
    // C[s][i] = kk a e^{g_ref - g_s}, K[s][i] = k e^{g_ref - g_s}, with e^{g_ref - g_s} = 1 / E[s][i].
    // Rows past the chunk's end are zero.
    auto phase2 = [&](int chunk, int lc, const float *eref) {
        {   // B_G: thread = row t, channels 4 cq .. 4 cq + 3 and 32 + 4 cq .. 32 + 4 cq + 3, so that
            // each 16-byte access of a quarter-warp (one row) covers 8 distinct bank groups.  A
            // warp takes rows b, b + 4, b + 1, b + 5 in its four quarters: the two rows of a
            // half-warp (its 8-byte tile reads) differ by 4, so their 64 bytes each lie in the
            // two complementary halves of the 128-byte swizzle pattern.
            const int wq = tid >> 5, jq = (tid >> 3) & 3;
            const int t = 8 * (wq >> 1) + 2 * (wq & 1) + 4 * (jq & 1) + (jq >> 1), cq = tid & 7;
            unsigned char *BG = sm + SM_BG;
            uint4 cw[2], kw[2];
            if (t < lc) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c4 = 4 * cq + 32 * h;
                    const float4 kkv = in4(rkk, p.kk, chunk, t, c4), av = in4(ra, p.a, chunk, t, c4),
                                 kv = in4(rk, p.k, chunk, t, c4);
                    const float4 e = *reinterpret_cast<const float4 *>(E + eidx(t, c4));
                    const float2 e0 = make_float2(rcp(e.x), rcp(e.y)), e1 = make_float2(rcp(e.z), rcp(e.w));
                    const float2 c0 = __fmul2_rn(__fmul2_rn(make_float2(kkv.x, kkv.y), make_float2(av.x, av.y)), e0);
                    const float2 c1 = __fmul2_rn(__fmul2_rn(make_float2(kkv.z, kkv.w), make_float2(av.z, av.w)), e1);
                    const float2 k0 = __fmul2_rn(make_float2(kv.x, kv.y), e0);
                    const float2 k1 = __fmul2_rn(make_float2(kv.z, kv.w), e1);
                    cw[h] = make_uint4(to_tf32(c0.x), to_tf32(c0.y), to_tf32(c1.x), to_tf32(c1.y));
                    kw[h] = make_uint4(to_tf32(k0.x), to_tf32(k0.y), to_tf32(k1.x), to_tf32(k1.y));
                }
            } else {
                cw[0] = cw[1] = kw[0] = kw[1] = make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                *reinterpret_cast<uint4 *>(BG + sw128_off(t, 4 * cq + 32 * h, 128)) = cw[h];
                *reinterpret_cast<uint4 *>(BG + sw128_off(64 + t, 4 * cq + 32 * h, 128)) = kw[h];
            }
        }
        {   // A_G: thread = TMEM lane m (row t of R, or of Q for m >= 64), channels 16 cg ..
            const bool rrow = m < 64;
            const int t = rrow ? m : m - 64;
            const int i0 = 16 * cg;
            uint32_t wds[16];
            if (t < lc) {
                float x[16];
                in8(rrow ? rr : rkk, rrow ? p.r : p.kk, chunk, t, i0, x);
                in8(rrow ? rr : rkk, rrow ? p.r : p.kk, chunk, t, i0 + 8, x + 8);
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    float4 e;
                    if (rrow) {
                        e = *reinterpret_cast<const float4 *>(E + eidx(t, i0 + j));
                    } else if (t > 0) {
                        e = *reinterpret_cast<const float4 *>(E + eidx(t - 1, i0 + j));
                    } else {
                        const float4 er = *reinterpret_cast<const float4 *>(eref + i0 + j);
                        e = make_float4(rcp(er.x), rcp(er.y), rcp(er.z), rcp(er.w));
                    }
                    const float2 p0 = __fmul2_rn(make_float2(x[j], x[j + 1]), make_float2(e.x, e.y));
                    const float2 p1 = __fmul2_rn(make_float2(x[j + 2], x[j + 3]), make_float2(e.z, e.w));
                    wds[j] = to_tf32(p0.x);
                    wds[j + 1] = to_tf32(p0.y);
                    wds[j + 2] = to_tf32(p1.x);
                    wds[j + 3] = to_tf32(p1.y);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) wds[j] = 0u;
            }
            tmem_st16(tmem + lane_off + kColAG + i0, wds);
        }
    };

    // V^T into B_chain (K 64..127)
    // Thread: columns j, j+1 (j even) of tokens s0 .. s0+3.  Half the lanes store row j first,
    // half row j+1, so each quarter-warp's 16-byte stores land in 8 distinct bank groups.
    auto write_vt = [&](int chunk, int lc) {
        if (kind == kItemTransfer) lc = 0;  // v = 0
        const int j = 2 * (tid & 31), s0 = 4 * (tid >> 5);
        float a0[4], a1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = s0 + e < lc ? in2(rv, p.v, chunk, s0 + e, j) : make_float2(0.f, 0.f);
            a0[e] = x.x;
            a1[e] = x.y;
        }
        const bool odd_first = (tid >> 2) & 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const bool odd = (h == 0) == odd_first;
            st_tf32x4(sm + SM_BC + sw128_off(j + (odd ? 1 : 0), 64 + s0, 64), odd ? a1[0] : a0[0], odd ? a1[1] : a0[1],
                      odd ? a1[2] : a0[2], odd ? a1[3] : a0[3]);
        }
    };

    // Gram product G = [R ; Q] [C ; K]^T.  The lower halves of A_X and of the base take
    // [C^T | K^T] (copied in phase 4): Cb^T and Kb^T without their row factor
    // e^{g_C - g_ref}[i] (Cb^T[i][s] = e^{g_C - g_ref}[i] C[s][i]).  That factor multiplies
    // every lower row of D's operands, so it is applied to the state rows of D instead.
    auto issue_gram = [&]() {
#pragma unroll
        for (int kq = 0; kq < 8; ++kq)
            mma_tf32_tmem_a(tmem + kColG, tmem + kColAG + 8 * kq,
                            sdesc_sw128(sbase + SM_BG + (kq >> 2) * 128 * 128 + (kq & 3) * 32),
                            idesc_tf32(128, 128), kq > 0);
    };

    bool alive = true;
    if (warp == kThreads / 32) {
        // ======== the MMA warp: one lane issues every tensor-core product, in
        // the order the workers hand the operands over, and every TMA copy, so
        // operand staging never waits for an issue.
        if (lane == 0) {
            uint32_t ip = 0;
            int last_load = nchunks > 1 ? 1 : 0;  // the last chunk whose tiles were requested
            auto ready = [&](uint32_t rdy, uint32_t parity) {
                const bool ok = mbar_wait_bounded(rdy, parity, kMaxPolls);
                tc_fence_after_sync();
                return ok;
            };
            auto wait_own = [&]() {  // the MMA warp's own wait on products it chains
                const bool ok = mbar_wait_bounded(bar_i, ip, kMaxPolls);
                ip ^= 1u;
                tc_fence_after_sync();
                return ok;
            };
            bool ok = ready(rdy_g, 0);  // chunk 0: Gram operands
            if (ok) {
                issue_gram();
                mma_commit(bar_g);
            }
            for (int c = 0; c < nchunks && ok; ++c) {
                const bool has_next = c + 1 < nchunks;
                const uint32_t par = static_cast<uint32_t>(c & 1);
                // W = [Q | L_k] [S0' ; V] over G's columns 0..63 (rows 0..63 of that product are
                // not used): as soon as G is read and L_k masked in place
                if (!(ok = ready(rdy_w, par))) break;
#pragma unroll
                for (int kq = 0; kq < 16; ++kq)
                    mma_tf32_tmem_a(tmem + kColG, tmem + (kq < 8 ? kColAG + 8 * kq : kColG + 64 + 8 * (kq - 8)),
                                    sdesc_sw128(sbase + SM_BC + (kq >> 2) * 64 * 128 + (kq & 3) * 32),
                                    idesc_tf32(128, 64), kq > 0);
                mma_commit(bar_w);
                // D = base [S0' ; V] as soon as the base is written (it needs no T either), so that
                // only X and D -= X W follow the T halves on the tensor core
                if (!(ok = ready(rdy_b, par))) break;
#pragma unroll
                for (int kq = 0; kq < 16; ++kq)
                    mma_tf32_tmem_a(tmem + kColD, tmem + kColAC + 8 * kq,
                                    sdesc_sw128(sbase + SM_BC + (kq >> 2) * 64 * 128 + (kq & 3) * 32),
                                    idesc_tf32(128, 64), kq > 0);
                // X = [M_c ; Cb^T] T in three products:
                //   X_R = B_R T_B -> X[:, 32:64);  B_L -= X_R L_BA (in place);  X_L = B_L T_A -> X[:, 0:32)
                if (!(ok = ready(rdy_x, par))) break;
#pragma unroll
                for (int kq = 0; kq < 4; ++kq)
                    mma_tf32_tmem_a(tmem + kColX + 32, tmem + kColAX + 32 + 8 * kq,
                                    sdesc_sw128(sbase + SM_BX + kq * 32), idesc_tf32(128, 32), kq > 0);
                mma_commit(bar_i);
                if (!(ok = wait_own())) break;
#pragma unroll
                for (int kq = 0; kq < 4; ++kq)
                    mma_tf32_tmem_a(tmem + kColAX, tmem + kColX + 32 + 8 * kq,
                                    sdesc_sw128(sbase + SM_BX + 4096 + kq * 32),
                                    idesc_tf32(128, 32) | kIdescNegateA, 1);
                mma_commit(bar_i);
                if (!(ok = wait_own())) break;
#pragma unroll
                for (int kq = 0; kq < 4; ++kq)
                    mma_tf32_tmem_a(tmem + kColX, tmem + kColAX + 8 * kq, sdesc_sw128(sbase + SM_BX + 8192 + kq * 32),
                                    idesc_tf32(128, 32), kq > 0);
                mma_commit(bar_i);
                if (!(ok = wait_own())) break;
                // D -= X W  (negated A, accumulating onto base [S0' ; V])
#pragma unroll
                for (int kq = 0; kq < 8; ++kq)
                    mma_tf32_tmem_a(tmem + kColD, tmem + kColX + 8 * kq,
                                    sdesc_sw128(sbase + SM_BY + (kq >> 2) * 64 * 128 + (kq & 3) * 32),
                                    idesc_tf32(128, 64) | kIdescNegateA, 1);
                // the previous chunk's output stores have read the staging tile, so D's completion
                // also tells the workers that they may stage this chunk's outputs
                bulk_wait_read<0>();
                mma_commit(bar_d);
                if (has_next) {  // the next chunk's Gram product
                    if (!(ok = ready(rdy_g, static_cast<uint32_t>((c + 1) & 1)))) break;
                    issue_gram();
                    mma_commit(bar_g);
                }
                // the workers have staged this chunk's outputs and consumed chunk c + 1's tiles
                if (!(ok = ready(rdy_t, par))) break;
                if (chunk_len(c) == kC) {
                    const int t0 = bos + (c_begin + c) * kC;
                    if (to_scratch) {
                        tma_store_2d(&maps.ohat, 0, ohat_row + c * kC, sbase + SM_TS);
                        tma_store_2d(&maps.ohat, 32, ohat_row + c * kC, sbase + SM_TS + 8192);
                    } else if (bf16_out) {
                        tma_store_2d(&maps.o, h * 64, t0, sbase + SM_TS);
                    } else {
                        tma_store_2d(&maps.o, h * 64, t0, sbase + SM_TS);
                        tma_store_2d(&maps.o, h * 64 + 32, t0, sbase + SM_TS + 8192);
                    }
                    bulk_commit();
                }
                if (c + 2 < nchunks) {
                    issue_tma(c + 2);
                    last_load = c + 2;
                }
            }
            if (!ok) report(p.status, kDevTimeout);
            bulk_wait<0>();  // every output store has completed
            // the last input load has landed before the CTA's shared memory goes away
            mbar_wait_bounded(bar_tma, static_cast<uint32_t>(last_load & 1), kMaxPolls);
        }
    } else {
    // ======== the 512 worker threads
    // ---- prologue: chunk 0 up to its Gram product
    if (tid == 0) issue_tma(0);
    alive = wait_uniform(bar_tma, 0, p.status);
    if (alive) {
        phase1(chunk_len(0), 0);
        wsync();
        // B_chain rows j, K 0..63 <- e^{g_ref}[i] S0[i][j]
        if (state_thread) {
            const float er = EREF[si];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                *reinterpret_cast<uint32_t *>(sm + SM_BC + sw128_off(16 * cg + j, si, 64)) = to_tf32(s[j] * er);
        }
        phase2(0, chunk_len(0), EREF);
        write_vt(0, chunk_len(0));
        handoff(rdy_g);
        if (tid == 0 && nchunks > 1) issue_tma(1);  // chunk 0's tiles are no longer read
        alive = wait_uniform(bar_g, 0, p.status);
        tc_fence_after_sync();
    }

    for (int c = 0; c < nchunks && alive; ++c) {
        const int t0 = bos + (c_begin + c) * kC;
        const int lc = chunk_len(c);
        const bool has_next = c + 1 < nchunks;
        const uint32_t par = static_cast<uint32_t>(c & 1);

        // ---- phase 3: read G.  M_c (masked) -> A_X rows t, which with Cb^T below them
        // (phase 4) form A_X = [M_c ; Cb^T]; M_k (masked) -> the base's rows t, K 64..;
        // L_c^T -> LT; L_k masked in place (G columns 64..127, rows 64..127: W's A operand
        // beside A_G's Q), 16 + 16 columns per lower-lane warp.  The two warps that compute
        // the T halves (0, 1) take no part: the lower-lane warps signal them as soon as L_c^T
        // is written (named barrier 2: 256 arrivals + their 64), so the inverse starts while
        // the rest of this phase runs, and warps 12, 13 take their share of M_c.  The others
        // finish the phase on named barrier 3 (448 threads) and hand W's operands over.
        if (q < 2) {
            if (warp >= 2) {
#pragma unroll 1
                for (int pass = 0; pass < (cg == 3 ? 2 : 1); ++pass) {
                    const int g = pass ? 0 : cg;  // warps 12, 13: M_k columns 32..63, then M_c 0..31
                    uint32_t wds[32];
                    const int gcol = (g < 2 ? 0 : 64) + 32 * (g & 1);  // M_c | M_k
                    const int s0 = 32 * (g & 1);
                    const int t = m;
                    float v[32];
                    tmem_ld32(tmem + lane_off + kColG + gcol, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) wds[j] = to_tf32(s0 + j <= t ? v[j] : 0.f);
                    tmem_st32_issue(tmem + lane_off + (gcol < 64 ? kColAX : kColAC) + gcol, wds);
                    tmem_wait_st();
                }
            }
        } else {
            const int t = m - 64, s0 = 16 * cg;
            float v[16];
            tmem_ld16(tmem + lane_off + kColG + s0, v);
            float *LTw = reinterpret_cast<float *>(sm + SM_LC);  // L_c^T: LT[s][t] = L_c[t][s]
#pragma unroll
            for (int j = 0; j < 16; ++j) LTw[(s0 + j) * kLd + t] = s0 + j < t ? v[j] : 0.f;
            named_arrive<2, 256 + 64>();  // -> the T halves
            tmem_ld16(tmem + lane_off + kColG + 64 + s0, v);
            uint32_t lw[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) lw[j] = to_tf32(s0 + j < t ? v[j] : 0.f);
            tmem_st16(tmem + lane_off + kColG + 64 + s0, lw);
        }
        if (warp < 2) {
            named_sync<2, 256 + 64>();  // L_c^T written
        } else {
            fence_proxy_async_smem();
            tc_fence_before_sync();
            named_sync<3, kThreads - 64>();
            tc_fence_after_sync();
            if (tid == 64) mbar_arrive(rdy_w);  // -> W = [Q | L_k] [S0' ; V]
        }

        // ---- phase 4: the two 32x32 diagonal halves of T = (I + L_c)^{-1}, in fp32, one warp
        // each: T_A = (I + L_AA)^{-1} (warp 0), T_B = (I + L_BB)^{-1} (warp 1).  Within a half
        // [T_00 0 ; T_10 T_11]: the 16x16 diagonal blocks by right-looking substitution (lane
        // = column; lanes 0..15 the first block, 16..31 the second), then T_10 = -T_11 (L_10 T_00)
        // with rows split between the two half-warps.  The off-diagonal half
        // T_BA = -T_B L_BA T_A is never formed: with [M_c ; Cb^T] = [B_L | B_R],
        //   X_R = B_R T_B,   X_L = (B_L - X_R L_BA) T_A
        // are three small MMAs.  Their B operands T_B^T, L_BA^T, T_A^T go to B_X
        // (B[n][k] = M[k][n]); the warps of the other two sub-partitions (warp % 4 = 2, 3)
        // meanwhile copy [C^T | K^T], stage L_BA^T and, once W is complete, W^T, so the two
        // inverse warps issue unhindered, and warps 4, 5, 8, 9 copy R into the base's S0
        // block.  With that, every operand of X, D = base [S0' ; V] and D -= X W is in place
        // at the end of this phase: the MMA warp runs them without another handoff while the
        // workers go on to the next chunk.
        {
            const float *LT = reinterpret_cast<const float *>(sm + SM_LC);
            if (warp < 2) {
                const int o = 32 * warp, hb = lane >> 4, j = lane & 15, ob = o + 16 * hb;
                float x[16];  // column j of this lane's diagonal block of T
#pragma unroll
                for (int t = 0; t < 16; ++t) x[t] = (t == j) ? 1.f : 0.f;
#pragma unroll
                for (int u = 0; u < 15; ++u) {
                    const float *lrow = LT + (ob + u) * kLd + ob;  // L[ob + t][ob + u], t = 0..15
#pragma unroll
                    for (int t4 = (u + 1) & ~3; t4 < 16; t4 += 4) {
                        const float4 l = *reinterpret_cast<const float4 *>(lrow + t4);
                        if (t4 + 0 > u) x[t4 + 0] = fmaf(-l.x, x[u], x[t4 + 0]);
                        if (t4 + 1 > u) x[t4 + 1] = fmaf(-l.y, x[u], x[t4 + 1]);
                        if (t4 + 2 > u) x[t4 + 2] = fmaf(-l.z, x[u], x[t4 + 2]);
                        if (t4 + 3 > u) x[t4 + 3] = fmaf(-l.w, x[u], x[t4 + 3]);
                    }
                }
                // Y = L_10 T_00, column j, rows 8 hb .. 8 hb + 7 (L_10[r][u] = L[o + 16 + r][o + u])
                float y[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) y[r] = 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float xa = __shfl_sync(0xffffffffu, x[u], j);  // T_00[u][j]
                    const float *lr = LT + (o + u) * kLd + o + 16 + 8 * hb;
                    const float4 l0 = *reinterpret_cast<const float4 *>(lr);
                    const float4 l1 = *reinterpret_cast<const float4 *>(lr + 4);
                    y[0] = fmaf(l0.x, xa, y[0]); y[1] = fmaf(l0.y, xa, y[1]);
                    y[2] = fmaf(l0.z, xa, y[2]); y[3] = fmaf(l0.w, xa, y[3]);
                    y[4] = fmaf(l1.x, xa, y[4]); y[5] = fmaf(l1.y, xa, y[5]);
                    y[6] = fmaf(l1.z, xa, y[6]); y[7] = fmaf(l1.w, xa, y[7]);
                }
                // T_10 = -T_11 Y, column j, rows 8 hb .. 8 hb + 7.  T_11 goes through this warp's
                // scratch (row-major 16 x 16, exact zeros above the diagonal).
                float *T11 = reinterpret_cast<float *>(sm + SM_XS) + warp * 256;
                if (hb) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) T11[r * 16 + j] = x[r];
                }
                float yv[16];  // Y[v][j], v = 0..15 (rows 8..15 are only needed, and only read, by hb = 1)
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    yv[v] = __shfl_sync(0xffffffffu, y[v], j);
                    yv[8 + v] = y[v];
                }
                __syncwarp();
                float z[8];
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const float *tr = T11 + (8 * hb + rr) * 16;
                    float acc = 0.f;
#pragma unroll
                    for (int v4 = 0; v4 < 16; v4 += 4) {
                        const float4 tv = *reinterpret_cast<const float4 *>(tr + v4);
                        acc = fmaf(tv.x, yv[v4], acc);
                        acc = fmaf(tv.y, yv[v4 + 1], acc);
                        acc = fmaf(tv.z, yv[v4 + 2], acc);
                        acc = fmaf(tv.w, yv[v4 + 3], acc);
                    }
                    z[rr] = -acc;
                }
                // B_X rows: row n = column n of the half's T
                unsigned char *dst = sm + SM_BX + (warp == 0 ? 8192 : 0);
                if (hb == 0) {
#pragma unroll
                    for (int k0 = 0; k0 < 16; k0 += 4) st_tf32x4(dst + sw128_off(j, k0, 32), x[k0], x[k0 + 1], x[k0 + 2], x[k0 + 3]);
                    st_tf32x4(dst + sw128_off(j, 16, 32), z[0], z[1], z[2], z[3]);
                    st_tf32x4(dst + sw128_off(j, 20, 32), z[4], z[5], z[6], z[7]);
                } else {
                    st_tf32x4(dst + sw128_off(j, 24, 32), z[0], z[1], z[2], z[3]);
                    st_tf32x4(dst + sw128_off(j, 28, 32), z[4], z[5], z[6], z[7]);
#pragma unroll
                    for (int k0 = 0; k0 < 16; k0 += 4) {
                        *reinterpret_cast<uint4 *>(dst + sw128_off(16 + j, k0, 32)) = make_uint4(0u, 0u, 0u, 0u);
                        st_tf32x4(dst + sw128_off(16 + j, 16 + k0, 32), x[k0], x[k0 + 1], x[k0 + 2], x[k0 + 3]);
                    }
                }
            } else if (!(warp & 2)) {
                // warps 4, 5 and 8, 9: the base's R block (this chunk's Gram A operand, upper
                // lanes) into the base's S0 columns
                if (cg < 3) {
                    const int c0 = 32 * (cg - 1);
                    float v[32];
                    uint32_t wds[32];
                    tmem_ld32(tmem + lane_off + kColAG + c0, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) wds[j] = __float_as_uint(v[j]);
                    tmem_st32_issue(tmem + lane_off + kColAC + c0, wds);
                    tmem_wait_st();
                }
                tc_fence_before_sync();
                named_sync<3, kThreads - 64>();  // the base is written
            } else {
                const int sidx = (((warp >> 2) << 1) | (warp & 1)) * 32 + lane;
                {   // [C^T | K^T] into A_X and base lanes 64..127 (row i = m - 64, columns s = 16 cg ..):
                    // the tf32 words of B_G with the rounding bits cleared, i.e. exactly the
                    // product of the identity with B_G
                    const int i = m - 64;
                    uint32_t cw[16], kw[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s_ = 16 * cg + j;
                        cw[j] = *reinterpret_cast<const uint32_t *>(sm + SM_BG + sw128_off(s_, i, 128)) & 0xffffe000u;
                        kw[j] = *reinterpret_cast<const uint32_t *>(sm + SM_BG + sw128_off(64 + s_, i, 128)) & 0xffffe000u;
                    }
                    tmem_st16(tmem + lane_off + kColAX + 16 * cg, cw);
                    tmem_st16(tmem + lane_off + kColAC + 64 + 16 * cg, kw);
                }
                {   // the base's zero block below R
                    uint32_t z[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) z[j] = 0u;
                    tmem_st16(tmem + lane_off + kColAC + 16 * cg, z);
                }
                tc_fence_before_sync();
                named_sync<3, kThreads - 64>();  // the base is written
                if (tid == 64) {
                    tc_fence_after_sync();
                    mbar_arrive(rdy_b);  // -> D = base [S0' ; V]
                }
                {   // L_BA^T: B[n][k] = L_c[32 + k][n] = LT[n][32 + k]
                    const int n = sidx >> 3, k0 = 4 * (sidx & 7);
                    const float4 l = *reinterpret_cast<const float4 *>(LT + n * kLd + 32 + k0);
                    st_tf32x4(sm + SM_BX + 4096 + sw128_off(n, k0, 32), l.x, l.y, l.z, l.w);
                }
                {   // W^T into B_Y (B[n][t] = W[t][n]) once the product is complete.  A wait that
                    // runs out is reported; the block then stops at its next uniform wait.
                    if (!mbar_wait_bounded(bar_w, par, kMaxPolls)) report(p.status, kDevTimeout);
                    tc_fence_after_sync();
                    const int t = m - 64;
                    float v[16];
                    tmem_ld16(tmem + lane_off + kColG + 16 * cg, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        *reinterpret_cast<uint32_t *>(sm + SM_BY + sw128_off(16 * cg + j, t, 64)) = to_tf32(v[j]);
                }
            }
        }
        handoff(rdy_x);  // -> X = [M_c ; Cb^T] T

        // ---- next chunk, phases 1 and 2 (overlap the X and D products)
        if (has_next) {
            if (!wait_uniform(bar_tma, static_cast<uint32_t>((c + 1) & 1), p.status)) { alive = false; break; }
            phase1(chunk_len(c + 1), (c + 1) & 1);
            wsync();
            phase2(c + 1, chunk_len(c + 1), EREF + ((c + 1) & 1) * 64);
            handoff(rdy_g);  // -> the next chunk's Gram products
        }
        if (!wait_uniform(bar_d, par, p.status)) { alive = false; break; }
        tc_fence_after_sync();

        // ---- phase 5: outputs, the state update, the next chunk's V^T
        {
            float v[16];
            tmem_ld16(tmem + lane_off + kColD + 16 * cg, v);
            if (q < 2) {
                const int t = m;
                if (bf16_out) {
                    // bf16 output: row t's 16 columns as two 16-byte words, staged (full chunk) in
                    // one 64 x 64 box of T's scratch (128-byte swizzle) for one TMA store below
                    uint4 wv[2];
#pragma unroll
                    for (int hw = 0; hw < 2; ++hw) {
                        uint32_t pk[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * hw + 2 * j], v[8 * hw + 2 * j + 1]);
                            pk[j] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        wv[hw] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                    if (lc == kC) {
                        unsigned char *row = sm + SM_TS + t * 128;
                        *reinterpret_cast<uint4 *>(row + (((2 * cg) ^ (t & 7)) << 4)) = wv[0];
                        *reinterpret_cast<uint4 *>(row + (((2 * cg + 1) ^ (t & 7)) << 4)) = wv[1];
                    } else if (t < lc) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + (t0 + t) * tok_stride +
                                                               h * 64 + 16 * cg);
                        dst[0] = wv[0];
                        dst[1] = wv[1];
                    }
                } else if (lc == kC) {
                    // full chunk: stage row t in T's scratch as two 64 x 32 boxes (128-byte
                    // swizzle), written out below by two TMA stores
                    unsigned char *box = sm + SM_TS + (cg >> 1) * 8192 + t * 128;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<float4 *>(box + (((4 * (cg & 1) + j) ^ (t & 7)) << 4)) =
                            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                } else if (t < lc) {
                    float4 *dst = reinterpret_cast<float4 *>(
                        to_scratch ? plan.ohat + (static_cast<long long>(ohat_row) + c * kC + t) * 64 + 16 * cg
                                              : static_cast<float *>(p.o) + (t0 + t) * tok_stride + h * 64 + 16 * cg);
#pragma unroll
                    for (int j = 0; j < 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
            } else {
                const float decay = GC[(c & 1) * 64 + si], rowf = E63[(c & 1) * 64 + si];
                const float ern = has_next ? EREF[((c + 1) & 1) * 64 + si] : 1.f;  // e^{g_ref} of the next chunk
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    s[j] = fmaf(decay, s[j], rowf * v[j]);
                    *reinterpret_cast<uint32_t *>(sm + SM_BC + sw128_off(16 * cg + j, si, 64)) = to_tf32(s[j] * ern);
                }
            }
            if (has_next) write_vt(c + 1, chunk_len(c + 1));
        }
        sync_for_mma();
        if (tid == 0) mbar_arrive(rdy_t);  // -> the output stores and the tiles of chunk c + 2
        if (has_next) {
            if (!wait_uniform(bar_g, static_cast<uint32_t>((c + 1) & 1), p.status)) { alive = false; break; }
            tc_fence_after_sync();
        }
    }

    // the final state: into a tail-split slot (fp32) or the caller's final_state (state_dtype)
    if (alive && state_thread && (slot >= 0 || p.final_state)) {
        void *fdst = slot >= 0 ? static_cast<void *>(plan.slots + static_cast<long long>(slot) * 4096) : p.final_state;
        const wkv7_dtype fdt = slot >= 0 ? WKV7_F32 : p.state_dtype;
        const long long fbase = (slot >= 0 ? 0 : sslot) + si * 64 + 16 * cg;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            store_state4(fdst, fdt, fbase + 4 * j, make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]));
    }
    }  // workers
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- scheduling

// Longest-first order of the sequences: order[rank] = sequence index, by
// descending length, ties by index.  One CTA sorts (key, index) pairs with a
// bitonic network in shared memory.  Blocks of the prefill kernel are handed
// out in blockIdx order as SMs free up, so launching the longest pairs first
// keeps a long sequence from starting last and stretching the tail.
constexpr int kOrderThreads = 1024;
constexpr int kMaxOrdered = 4096;  // sequences sorted on the device; more keep input order

__global__ void __launch_bounds__(kOrderThreads)
wkv7_prefill_order_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ lens, int num_seqs,
                          int32_t *__restrict__ order) {
    __shared__ unsigned long long key[kMaxOrdered];
    int n2 = 1;
    while (n2 < num_seqs) n2 <<= 1;
    for (int i = threadIdx.x; i < n2; i += kOrderThreads) {
        unsigned long long k = ~0ull;  // padding sorts last
        if (i < num_seqs) {
            const int len = max(0, lens ? lens[i] : cu[i + 1] - cu[i]);
            // ascending sort of (~len, index) = descending length, then index
            k = (static_cast<unsigned long long>(0x7fffffff - len) << 32) | static_cast<unsigned>(i);
        }
        key[i] = k;
    }
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n2; i += kOrderThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    const unsigned long long a = key[i], b = key[j];
                    if ((a > b) == up) {
                        key[i] = b;
                        key[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < num_seqs; i += kOrderThreads) order[i] = static_cast<int32_t>(key[i] & 0xffffffffu);
}

// ---------------------------------------------------------------- tail-split fix-up

constexpr int kFixThreads = 256;

// 64x64 products in fp32 on 256 threads, each owning a 4x4 tile (rows 4 tr.., columns
// 4 tc..): acc += A B with A held transposed (At[k][row], stride kLdT) and B row-major
// (stride 64), both in shared memory; per k one 16-byte load of each gives 16 FMAs.
constexpr int kLdT = 68;
// The inner product runs on paired fp32 FMAs (two lanes of a float2 per instruction;
// each element is the same single fmaf as before).
__device__ __forceinline__ void mm64_tile(const float *At, const float *B, int tr, int tc, float (&acc)[4][4]) {
    float2 acc2[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        acc2[r][0] = make_float2(acc[r][0], acc[r][1]);
        acc2[r][1] = make_float2(acc[r][2], acc[r][3]);
    }
#pragma unroll 8
    for (int k = 0; k < 64; ++k) {
        const float4 a = *reinterpret_cast<const float4 *>(At + k * kLdT + 4 * tr);
        const float4 b = *reinterpret_cast<const float4 *>(B + k * 64 + 4 * tc);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float2 ar = make_float2(av[r], av[r]);
            acc2[r][0] = __ffma2_rn(ar, b01, acc2[r][0]);
            acc2[r][1] = __ffma2_rn(ar, b23, acc2[r][1]);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        acc[r][0] = acc2[r][0].x; acc[r][1] = acc2[r][0].y;
        acc[r][2] = acc2[r][1].x; acc[r][3] = acc2[r][1].y;
    }
}
// global row-major 64x64 fp32 -> shared, transposed (dst[k][row], stride kLdT)
__device__ __forceinline__ void load_t64(float *dst, const float *src) {
    for (int e = threadIdx.x; e < 1024; e += kFixThreads) {
        const float4 x = reinterpret_cast<const float4 *>(src)[e];
        const int row = e >> 4, k0 = 4 * (e & 15);
        dst[(k0 + 0) * kLdT + row] = x.x;
        dst[(k0 + 1) * kLdT + row] = x.y;
        dst[(k0 + 2) * kLdT + row] = x.z;
        dst[(k0 + 3) * kLdT + row] = x.w;
    }
}

// One CTA per split pair: the true state at every segment boundary, in order,
// S_in(j+1) = P(j) S_in(j) + S_part(j), written over S_part(j)'s slot; the
// last one is the pair's final state.  The products are a dependent chain, so
// the CTA is large (1024 threads, a 2 x 2 output tile each: rows 2 tr .., columns
// 2 tc ..) to keep each product short.
constexpr int kChainThreads = 1024;

__global__ void __launch_bounds__(kChainThreads)
wkv7_prefill_split_chain_kernel(const __grid_constant__ FixPlan fp, void *final_state, wkv7_dtype state_dtype, int H) {
    __shared__ __align__(16) float sin_[64 * 64];
    __shared__ __align__(16) float pt[64 * kLdT];  // P(j) transposed
    const FixPair &pr = fp.pair[blockIdx.x];
    const int tid = threadIdx.x, tr = tid >> 5, tc = tid & 31;
    const float4 *s0 = reinterpret_cast<const float4 *>(fp.slots + static_cast<long long>(pr.seg[0].slot_part) * 4096);
    reinterpret_cast<float4 *>(sin_)[tid] = s0[tid];  // 1024 float4 = the 64 x 64 state
    // this thread's float4 of P(j) and 2 x 2 tile of S_part(j), fetched one segment ahead
    auto fetch = [&](int j, float4 &x, float2 (&sp)[2]) {
        x = reinterpret_cast<const float4 *>(fp.slots + static_cast<long long>(pr.seg[j].slot_transfer) * 4096)[tid];
        const float *Sp = fp.slots + static_cast<long long>(pr.seg[j].slot_part) * 4096;
#pragma unroll
        for (int r = 0; r < 2; ++r) sp[r] = *reinterpret_cast<const float2 *>(Sp + (2 * tr + r) * 64 + 2 * tc);
    };
    float4 xn;
    float2 spn[2];
    if (pr.nseg > 1) fetch(1, xn, spn);
    for (int j = 1; j < pr.nseg; ++j) {
        {   // P(j) transposed into pt[k][row]: one float4 of a row per thread
            const int row = tid >> 4, k0 = 4 * (tid & 15);
            pt[(k0 + 0) * kLdT + row] = xn.x;
            pt[(k0 + 1) * kLdT + row] = xn.y;
            pt[(k0 + 2) * kLdT + row] = xn.z;
            pt[(k0 + 3) * kLdT + row] = xn.w;
        }
        float *Sp = fp.slots + static_cast<long long>(pr.seg[j].slot_part) * 4096;
        float2 acc[2] = {spn[0], spn[1]};
        if (j + 1 < pr.nseg) fetch(j + 1, xn, spn);  // lands during this product
        __syncthreads();  // P(j)^T and S_in(j) in shared memory
#pragma unroll 8
        for (int k = 0; k < 64; ++k) {
            const float2 a = *reinterpret_cast<const float2 *>(pt + k * kLdT + 2 * tr);
            const float2 bv = *reinterpret_cast<const float2 *>(sin_ + k * 64 + 2 * tc);
            acc[0] = __ffma2_rn(make_float2(a.x, a.x), bv, acc[0]);
            acc[1] = __ffma2_rn(make_float2(a.y, a.y), bv, acc[1]);
        }
        __syncthreads();  // every thread has read S_in(j) and P(j)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            *reinterpret_cast<float2 *>(sin_ + (2 * tr + r) * 64 + 2 * tc) = acc[r];
            *reinterpret_cast<float2 *>(Sp + (2 * tr + r) * 64 + 2 * tc) = acc[r];
        }
    }
    __syncthreads();
    if (final_state) {
        const long long base = (static_cast<long long>(pr.b) * H + pr.h) * 4096;
        store_state4(final_state, state_dtype, base + 4 * tid, reinterpret_cast<const float4 *>(sin_)[tid]);
    }
}

// Grid (chunks after a pair's first segment, split pairs): o_t += S_in(j)^T (P_t^T r_t)
// for every token of segment j >= 1, as the 64x64x64 product [P_t^T r_t]_t S_in(j).
__global__ void __launch_bounds__(kFixThreads)
wkv7_prefill_split_ofix_kernel(const __grid_constant__ FixPlan fp, PrefillArgs p) {
    __shared__ __align__(16) float sin_[64 * 64];
    __shared__ __align__(16) float oht[64 * kLdT];  // readout rows, transposed
    const FixPair &pr = fp.pair[blockIdx.y];
    const int chunk = pr.seg[1].c0 + static_cast<int>(blockIdx.x);
    int j = 1;
    while (j < pr.nseg && chunk >= pr.seg[j].c1) ++j;
    if (j >= pr.nseg) return;  // past this pair's last chunk
    const FixSeg &sg = pr.seg[j];
    const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;
    // S_in(j): the true state at the segment's start (segment 0's slot or, for j >= 2,
    // the chain kernel's result over S_part(j - 1))
    const float4 *Sin = reinterpret_cast<const float4 *>(fp.slots + static_cast<long long>(pr.seg[j - 1].slot_part) * 4096);
    for (int e = tid; e < 1024; e += kFixThreads) reinterpret_cast<float4 *>(sin_)[e] = Sin[e];
    load_t64(oht, fp.ohat + (static_cast<long long>(sg.ohat_row) + (chunk - sg.c0) * 64) * 64);
    int bos, eos;
    seq_bounds(p, pr.b, bos, eos);
    const int t0 = bos + chunk * 64;
    const int lc = min(64, eos - t0);
    const bool bf16 = p.o_dtype == WKV7_BF16;
    // the partial outputs this thread corrects (in o, fp32; or in the part item's fp32 rows when
    // o is bf16), fetched before the product so that their latency overlaps it
    float4 part[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = 4 * tr + r;
        part[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < lc) {
            const long long at = (static_cast<long long>(t0) + t) * p.H * 64 + pr.h * 64 + 4 * tc;
            part[r] = bf16 ? *reinterpret_cast<const float4 *>(
                                 fp.ohat + (static_cast<long long>(sg.opart_row) + (chunk - sg.c0) * 64 + t) * 64 + 4 * tc)
                           : *reinterpret_cast<const float4 *>(static_cast<float *>(p.o) + at);
        }
    }
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
    mm64_tile(oht, sin_, tr, tc, acc);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = 4 * tr + r;
        if (t < lc) {
            const long long at = (static_cast<long long>(t0) + t) * p.H * 64 + pr.h * 64 + 4 * tc;
            float4 v = part[r];
            v.x += acc[r][0];
            v.y += acc[r][1];
            v.z += acc[r][2];
            v.w += acc[r][3];
            if (bf16) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
                uint2 u;
                u.x = *reinterpret_cast<const uint32_t *>(&lo);
                u.y = *reinterpret_cast<const uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.o) + at) = u;
            } else {
                *reinterpret_cast<float4 *>(static_cast<float *>(p.o) + at) = v;
            }
        }
    }
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

// 2-D map over a packed [T_total, H*64] array with 64 x 64 boxes: bf16 tiles
// in the 128-byte swizzle layout, fp32 (w) tiles unswizzled.
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
               bf16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output [T_total, H*64] written as 64-row boxes of 128 bytes in the 128-byte swizzle layout:
// 32 fp32 or 64 bf16 columns.
bool make_out_map(CUtensorMap *map, void *base, int T_total, int H, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * 64, static_cast<cuuint64_t>(T_total)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 64 * esz};
    cuuint32_t box[2] = {bf16 ? 64u : 32u, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// fp32 [rows, 64] scratch of the transfer items' readouts, same boxes as the output.
bool make_ohat_map(CUtensorMap *map, float *base, long long rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {64 * 4};
    cuuint32_t box[2] = {32, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

constexpr size_t kSlotsBytes = static_cast<size_t>(kMaxSplitItems) * 4096 * sizeof(float);

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// The tail-split schedule (see SplitItem).  With P pairs on S SMs (one CTA per SM),
// the last r = P mod S pairs in schedule order (the shortest) would run alone in a
// last wave (split when 0 < r <= S/2 and r <= kMaxSplitPairs).  Each is cut into k
// segments, the first of about f0 of its chunks and the others equal (2k - 1
// items: the first segment, then a part and a transfer item per later segment).
// Items start in launch order as SMs free up, so (k, f0) is chosen from a model of that
// list schedule (a few integer operations per candidate, no search on the host's
// critical path): when 2k - 1 items per pair fit on the SMs at once the best is k equal
// segments; when they do not, a longer first segment lets the short items run in rounds
// beside it (r = 64 pairs of 512 chunks: k = 3, a first segment of 307 chunks, against
// 512 whole and 342 for a 2:1 cut).  Needs the
// host copy of cu_seqlens; returns false (whole pairs only) otherwise.
bool plan_split(const PrefillArgs &a, unsigned char *split_ws, size_t split_bytes, SplitPlan &plan, FixPlan &fix) {
    const long long P = static_cast<long long>(a.num_seqs) * a.H;
    plan.main_items = static_cast<int>(P);
    plan.n_items = 0;
    plan.slots = plan.ohat = nullptr;
    fix.n_pairs = fix.n_blocks = 0;
    int len0 = 0;
    if (!host_seq_len(a, 0, len0) || !split_ws || split_bytes < kSlotsBytes + 64 * 256) return false;
    // with a bf16 output the part items' outputs also go to fp32 scratch rows
    const int rows_per = a.o_dtype == WKV7_BF16 ? 2 : 1;
    const long long rows_cap = static_cast<long long>((split_bytes - kSlotsBytes) / 256) & ~63ll;
    const int S = sm_count();
    if (S <= 0) return false;
    const long long r = P % S;
    if (r == 0 || 2 * r > S || r > kMaxSplitPairs) return false;
    auto len = [&](int b) {
        int l = 0;
        host_seq_len(a, b, l);
        return l;
    };
    // the schedule's sequence order: the device order kernel's (descending length, ties by index)
    std::vector<int> ord(a.num_seqs);
    std::iota(ord.begin(), ord.end(), 0);
    if (a.order) std::stable_sort(ord.begin(), ord.end(), [&](int x, int y) { return len(x) > len(y); });
    struct Tail { int b, h, n; };
    std::vector<Tail> tail;
    for (long long bi = P - r; bi < P; ++bi) {
        const int b = ord[bi / a.H];
        tail.push_back({b, static_cast<int>(bi % a.H), (len(b) + kC - 1) / kC});
    }
    // segment j of a pair of n chunks cut into kp segments, the first of about f0 / 1000 of
    // them, the others equal: [bound(j), bound(j + 1)), every segment at least one chunk
    auto segs = [&](const Tail &t, int k) { return t.n > 32767 || t.n < 3 ? 1 : std::min(k, t.n / 2); };
    auto bound = [&](const Tail &t, int kp, int f0, int j) {
        if (j <= 0) return 0;
        if (j >= kp) return t.n;
        const int l0 = std::min(t.n - (kp - 1), std::max(1, (f0 * t.n + 500) / 1000));
        return l0 + (j - 1) * (t.n - l0) / (kp - 1);
    };
    // Candidates k = 2 .. kMaxSegs, each with the first-segment share f0 (per mille) that
    // balances the list schedule, and its length in chunks (-1: does not fit).  When every
    // item starts at once the segments are equal and the tail takes the longest one.  When
    // not, the first segments hold r SMs and the 2 (k - 1) r short items run in rounds on
    // the other S - r (a model of the longest pair: rounds x short = first segment).
    int nmax = 0;
    for (const Tail &t : tail) nmax = std::max(nmax, t.n);
    auto candidate = [&](int k, int &f0) -> long long {
        long long items = 0, rows = 0, nsplit = 0;
        for (const Tail &t : tail) items += segs(t, k) < 2 ? 1 : 2 * segs(t, k) - 1;
        if (items <= S) {
            f0 = 1000 / k;
        } else {
            const long long rounds = (items - r + (S - r) - 1) / (S - r);
            f0 = static_cast<int>((1000 * rounds) / (rounds + k - 1));
        }
        long long span = 0;
        for (const Tail &t : tail) {
            const int kp = segs(t, k);
            if (kp < 2) {
                span = std::max<long long>(span, t.n);
                continue;
            }
            ++nsplit;
            rows += static_cast<long long>(t.n - bound(t, kp, f0, 1)) * 64 * rows_per;
            span = std::max<long long>(span, bound(t, kp, f0, 1));
            if (items <= S)
                for (int j = 1; j < kp; ++j) span = std::max<long long>(span, bound(t, kp, f0, j + 1) - bound(t, kp, f0, j));
        }
        if (nsplit == 0 || items > kMaxSplitItems || rows > rows_cap) return -1;
        if (items > S) {  // the short items' rounds beside the first segments (longest pair)
            const Tail lp{0, 0, nmax};
            const int kp = segs(lp, k);
            if (kp >= 2) {
                const long long rounds = (items - r + (S - r) - 1) / (S - r);
                const long long short_len = (nmax - bound(lp, kp, f0, 1) + kp - 2) / (kp - 1);
                span = std::max(span, rounds * short_len);
            }
        }
        return span;
    };
    int best_k = 0, best_f = 0;
    long long best = -1;
    for (int k = 2; k <= kMaxSegs; ++k) {
        int f0 = 0;
        const long long m = candidate(k, f0);
        if (m >= 0 && (best < 0 || m < best)) {
            best = m;
            best_k = k;
            best_f = f0;
        }
    }
    if (best < 0) return false;
    {
        const int k = best_k, f0 = best_f;
        plan.main_items = static_cast<int>(P - r);
        plan.slots = fix.slots = reinterpret_cast<float *>(split_ws);
        plan.ohat = fix.ohat = reinterpret_cast<float *>(split_ws + kSlotsBytes);
        // items in dispatch order: whole tail pairs and first segments, then the rest
        int n = 0, slot = 0, blk = 0;
        long long row = 0;
        for (const Tail &t : tail) {
            const int pair = t.b * a.H + t.h, kp = segs(t, k);
            if (kp < 2) {
                plan.item[n++] = {pair, 0, static_cast<int16_t>(t.n), kItemWhole, -1, 0};
                continue;
            }
            FixPair &fp = fix.pair[fix.n_pairs++];
            fp.b = t.b;
            fp.h = t.h;
            fp.nseg = kp;
            FixSeg &sg = fp.seg[0];
            sg.c0 = 0;
            sg.c1 = static_cast<int16_t>(bound(t, kp, f0, 1));
            sg.slot_part = static_cast<int16_t>(slot);
            sg.slot_transfer = -1;
            sg.ohat_row = 0;
            sg.opart_row = 0;
            plan.item[n++] = {pair, sg.c0, sg.c1, kItemWhole, static_cast<int16_t>(slot++), 0};
        }
        for (int f = 0; f < fix.n_pairs; ++f) {
            FixPair &fp = fix.pair[f];
            const Tail t{fp.b, fp.h, (len(fp.b) + kC - 1) / kC};
            const int pair = fp.b * a.H + fp.h;
            for (int j = 1; j < fp.nseg; ++j) {
                FixSeg &sg = fp.seg[j];
                sg.c0 = static_cast<int16_t>(bound(t, fp.nseg, f0, j));
                sg.c1 = static_cast<int16_t>(bound(t, fp.nseg, f0, j + 1));
                sg.slot_part = static_cast<int16_t>(slot);
                sg.opart_row = 0;
                if (rows_per == 2) {
                    sg.opart_row = static_cast<int32_t>(row);
                    row += static_cast<long long>(sg.c1 - sg.c0) * 64;
                }
                plan.item[n++] = {pair, sg.c0, sg.c1, kItemPart, static_cast<int16_t>(slot++), sg.opart_row};
                sg.slot_transfer = static_cast<int16_t>(slot);
                sg.ohat_row = static_cast<int32_t>(row);
                plan.item[n++] = {pair, sg.c0, sg.c1, kItemTransfer, static_cast<int16_t>(slot++), static_cast<int32_t>(row)};
                row += static_cast<long long>(sg.c1 - sg.c0) * 64;
            }
            blk = std::max(blk, fp.seg[fp.nseg - 1].c1 - fp.seg[1].c0);
        }
        plan.n_items = n;
        fix.n_blocks = blk;
    }
    return true;
}

cudaError_t launch_chunked(const PrefillArgs &args, unsigned char *split_ws, size_t split_bytes, cudaStream_t stream) {
    TensorMaps maps;
    // bf16 inputs: swizzled 64 x 64 boxes staged in shared memory; fp32 inputs: plain 64 x 64
    // fp32 boxes, used only for the L2 prefetch
    const bool bf16_in = args.x_dtype == WKV7_BF16;
    if (!make_map(&maps.r, args.r, bf16_in, args.T_total, args.H) ||
        !make_map(&maps.k, args.k, bf16_in, args.T_total, args.H) ||
        !make_map(&maps.v, args.v, bf16_in, args.T_total, args.H) ||
        !make_map(&maps.kk, args.kk, bf16_in, args.T_total, args.H) ||
        !make_map(&maps.a, args.a, bf16_in, args.T_total, args.H) ||
        !make_map(&maps.w, args.w, false, args.T_total, args.H) || !make_out_map(&maps.o, args.o, args.T_total, args.H, args.o_dtype == WKV7_BF16))
        return cudaErrorInvalidValue;
    SplitPlan plan;
    FixPlan fix;
    const bool split = plan_split(args, split_ws, split_bytes, plan, fix);
    if (split && !make_ohat_map(&maps.ohat, plan.ohat, static_cast<long long>((split_bytes - kSlotsBytes) / 256) & ~63ll))
        return cudaErrorInvalidValue;
    static int attr_dev[2] = {-1, -1};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_dev[bf16_in] != dev) {
        e = cudaFuncSetAttribute(bf16_in ? wkv7_prefill_chunked_kernel<false> : wkv7_prefill_chunked_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_dev[bf16_in] = dev;
    }
    const unsigned grid = static_cast<unsigned>(plan.main_items + plan.n_items);
    if (bf16_in)
        wkv7_prefill_chunked_kernel<false><<<grid, kBlock, kSmemAlloc, stream>>>(args, maps, plan);
    else
        wkv7_prefill_chunked_kernel<true><<<grid, kBlock, kSmemAlloc, stream>>>(args, maps, plan);
    e = cudaGetLastError();
    if (e != cudaSuccess || !split) return e;
    wkv7_prefill_split_chain_kernel<<<fix.n_pairs, kChainThreads, 0, stream>>>(fix, args.final_state, args.state_dtype,
                                                                                args.H);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    wkv7_prefill_split_ofix_kernel<<<dim3(fix.n_blocks, fix.n_pairs), kFixThreads, 0, stream>>>(fix, args);
    return cudaGetLastError();
}

}  // namespace

// Workspace: [the longest-first order of the sequences (int32 per sequence, for
// batches of 2 .. kMaxOrdered sequences) | tail-split scratch: kMaxSplitItems
// state slots, then readout rows of 64 fp32 for up to min(T_total*H, 2^20)
// token-heads (none below 1024 tokens)].  Only the order part is required.
size_t prefill_workspace_min_bytes(int num_seqs) {
    if (num_seqs < 2 || num_seqs > kMaxOrdered) return 0;
    return (static_cast<size_t>(num_seqs) * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
}

size_t prefill_workspace_bytes(int num_seqs, int T_total, int H) {
    size_t bytes = prefill_workspace_min_bytes(num_seqs);
    if (T_total >= 1024 && num_seqs >= 1) {
        const long long rows = std::min<long long>(static_cast<long long>(T_total) * H, 1ll << 20) & ~63ll;
        bytes += kSlotsBytes + static_cast<size_t>(rows) * 256;
    }
    return bytes;
}

bool prefill_wants_order(const PrefillArgs &args) {
    if (args.num_seqs < 2 || args.num_seqs > kMaxOrdered || args.x_dtype == WKV7_F32) return false;
    int len0 = 0, len = 0;
    if (!host_seq_len(args, 0, len0)) return true;  // lengths unknown on the host: sort on the device
    for (int b = 1; b < args.num_seqs; ++b)
        if (host_seq_len(args, b, len) && len != len0) return true;
    return false;  // all lengths equal: the input order is already longest-first
}

cudaError_t launch_prefill_order(const PrefillArgs &args, int32_t *order, cudaStream_t stream) {
    wkv7_prefill_order_kernel<<<1, kOrderThreads, 0, stream>>>(args.cu_seqlens, args.lens, args.num_seqs, order);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs &args, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    const long long pairs = static_cast<long long>(args.num_seqs) * args.H;
    if (pairs <= 0) return cudaSuccess;
    const size_t state_bytes = static_cast<size_t>(pairs) * 4096 * state_elem_bytes(args.state_dtype);
    if (args.T_total == 0) {  // every sequence is empty: final = initial (or zeros)
        if (!args.final_state) return cudaSuccess;
        if (!args.initial_state) return cudaMemsetAsync(args.final_state, 0, state_bytes, stream);
        if (args.initial_state == args.final_state) return cudaSuccess;
        return cudaMemcpyAsync(args.final_state, args.initial_state, state_bytes, cudaMemcpyDeviceToDevice, stream);
    }
    // bf16 inputs (the prefill format) and fp32 inputs marked for tf32 contraction take the
    // chunked tensor-core kernel; plain fp32 inputs take the exact token-serial kernel.
    if (args.x_dtype == WKV7_BF16 || args.x_dtype == WKV7_TF32) {
        const size_t head = prefill_workspace_min_bytes(args.num_seqs);
        unsigned char *split_ws = workspace && workspace_bytes > head ? static_cast<unsigned char *>(workspace) + head : nullptr;
        return launch_chunked(args, split_ws, split_ws ? workspace_bytes - head : 0, stream);
    }
    return launch_prefill_scan(args, stream);
}

}  // namespace wkv7
