/*
 * wkv7.h -- C ABI of the WKV-7 recurrence on one NVIDIA GB300 (sm_103a).
 *
 * The operation (per head, head size N, state S = [K, V] = [N, N] fp32):
 *
 *     z   = kk^T S_old
 *     S   = diag(exp w) S_old - (kk .* a) z^T + k v^T
 *     o   = S^T r
 *
 * This is the per-head WKV7 update of the Core AI model zoo note
 * "Recurrent / linear-attention LLMs on Core AI", section 1 ("decode
 * recurrence lowers to standard ops"): decay and delta term both act on the
 * old state, the k v^T write follows, and the read-out sees the new state.
 * w is the log-decay (the decay factor is exp(w)); kk is used exactly as
 * given (the caller normalises it); a is a per-channel vector.  The state
 * layout [K, V] with the value channel contiguous is the recState layout of
 * section 2 of the same note.
 *
 * Conventions shared by every call:
 *   - Only N = 64 is supported (the head size of every RWKV-7 model the
 *     pages name); any other N returns WKV7_ERR_UNSUPPORTED.
 *   - All tensor pointers are DEVICE pointers owned by the caller and must be
 *     16-byte aligned (WKV7_ERR_ALIGNMENT otherwise).  The library allocates
 *     no memory and keeps no per-call state.
 *   - Every call is stream-ordered on `stream` (0 = legacy default stream)
 *     and returns without synchronising.  A launch failure returns
 *     WKV7_ERR_CUDA; errors found on the device (malformed cu_seqlens, an
 *     expired bounded wait) are recorded in a per-device status word that
 *     wkv7_check_device_status() reads and clears.
 *   - No call ever aborts, traps or asserts on the device; invalid arguments
 *     are rejected on the host before any launch.
 *   - All arithmetic is fp32 with fp32 state; decode inputs are fp32,
 *     prefill inputs r, k, v, kk, a may be bf16 (w is always fp32).
 */
#ifndef WKV7_H
#define WKV7_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define WKV7_API __attribute__((visibility("default")))
#else
#define WKV7_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WKV7_OK = 0,
    WKV7_ERR_INVALID_ARG = 1,  /* null pointer, bad size, malformed cu_seqlens, forbidden aliasing */
    WKV7_ERR_UNSUPPORTED = 2,  /* N != 64, unknown dtype */
    WKV7_ERR_ALIGNMENT = 3,    /* a tensor pointer is not 16-byte aligned */
    WKV7_ERR_CUDA = 4,         /* a CUDA runtime/launch error (see wkv7_last_cuda_error) */
    WKV7_ERR_TIMEOUT = 5,      /* a bounded device-side wait expired (device status) */
    WKV7_ERR_WORKSPACE = 6,    /* workspace missing or too small to hold the sequence order */
    WKV7_ERR_DEVICE_BOUNDS = 7 /* the device found an index out of range (device status) */
} wkv7_status;

typedef enum {
    WKV7_F32 = 0,
    WKV7_BF16 = 1,
    WKV7_F16 = 2,  /* IEEE half precision; accepted only where a call says so */
    WKV7_TF32 = 3  /* fp32 storage contracted at tf32 precision on the tensor cores;
                      accepted only where a call says so (the prefill inputs) */
} wkv7_dtype;

#define WKV7_HEAD_SIZE 64

/*
 * wkv7_step -- one decode token for B * H independent heads.
 *
 * The recurrent "step(id, state:)" of the SwiftRWKV inference page
 * ("Recurrent -- step(id, state:), one token at a time carrying RWKVState"),
 * restricted to the WKV part: the state is read and written in place.
 *
 *   r, w, k, v, kk, a : fp32 [B, H, N]      inputs of this token (w = log-decay)
 *   state             : fp32 [B, H, N, N]   [K][V], read and overwritten
 *   o                 : fp32 [B, H, N]      output o = S_new^T r
 *
 * B >= 0, H >= 1; B * H * N * N must fit in int64.  B == 0 is a no-op.
 * `state` must not overlap any input or `o` (WKV7_ERR_INVALID_ARG).
 */
WKV7_API wkv7_status wkv7_step(int B, int H, int N,
                      const float *r, const float *w, const float *k,
                      const float *v, const float *kk, const float *a,
                      float *state, float *o, cudaStream_t stream);

/*
 * wkv7_step_state -- wkv7_step with the state stored in state_dtype: WKV7_F32
 * (exactly wkv7_step_cast), WKV7_F16 or WKV7_BF16.  A 16-bit state is widened
 * to fp32 on load, the update and the read-out run in fp32 as in wkv7_step,
 * and the new state is rounded to nearest even when it is stored back in
 * place.  The Core AI model zoo note (section 5, "Parity gate + tokenizer")
 * runs an fp16 export with fp16 state arrays; a 16-bit state halves the state
 * traffic, which is 95% of a decode step's bytes.  Each step rounds the state
 * once, so over many steps it drifts from an fp32-state run by about one
 * 16-bit rounding per step (relative 2^-11 for fp16, 2^-8 for bf16), damped by
 * the decay.
 *
 *   r, w, k, v, kk, a : fp32 [B, H, N]
 *   state             : state_dtype [B, H, N, N], read and overwritten
 *   o                 : o_dtype [B, H, N] (WKV7_F32 or WKV7_BF16)
 *
 * Same rules as wkv7_step (sizes, alignment, no overlap of state with any
 * other argument) with the byte sizes of the chosen types.
 */
WKV7_API wkv7_status wkv7_step_state(int B, int H, int N,
                      const float *r, const float *w, const float *k,
                      const float *v, const float *kk, const float *a,
                      void *state, wkv7_dtype state_dtype, void *o, wkv7_dtype o_dtype,
                      cudaStream_t stream);

/*
 * The time-mix tail after WKV, per row and head of N channels:
 *
 *     y = (GroupNorm_head(o) * ln_w + ln_b + (sum_i r_i k_i r_k_i) v) * g
 *
 * GroupNorm_head(o)_j = (o_j - mean(o)) / sqrt(var(o) + eps) over the head's N
 * channels (var = the mean squared deviation).  The SwiftRWKV inference page
 * names these parts of the tail ("group norm, bonus, gate"; fused with the
 * recurrent step's kernels in "What the decode path is made of" and run over
 * the B*T rows of a prompt in the fp32-stream prefill notes); the RWKV-X page
 * lists r_k as a per-head weight [n_head, head_size].  The pages print no
 * formula and no eps: the group is one head, eps is the caller's, ln_w and
 * ln_b are per channel of each head, the bonus is added after the norm's
 * affine part and the gate multiplies the sum.
 *
 * wkv7_step_tail -- wkv7_step with the tail fused into the same kernel.
 *
 *   r, w, k, v, kk, a, state : as wkv7_step
 *   o                 : fp32 [B, H, N] (the WKV output) or NULL (not written)
 *   r_k, ln_w, ln_b   : fp32 [H, N]    per-layer parameters
 *   g                 : fp32 [B, H, N] the gate of this token
 *   eps               : the norm's epsilon, finite and >= 0
 *   y                 : fp32 [B, H, N] output
 *
 * All pointers are device pointers, 16-byte aligned.  `state` overlaps nothing
 * else; o and y overlap no input, no parameter and not each other
 * (WKV7_ERR_INVALID_ARG).
 */
WKV7_API wkv7_status wkv7_step_tail(int B, int H, int N,
                      const float *r, const float *w, const float *k,
                      const float *v, const float *kk, const float *a,
                      float *state, float *o,
                      const float *r_k, const float *ln_w, const float *ln_b,
                      const float *g, float eps, float *y, cudaStream_t stream);

/*
 * wkv7_tmix_tail -- the tail over n_rows packed rows, e.g. the outputs of
 * wkv7_prefill ([T_total, H, N]).
 *
 *   o               : fp32 [n_rows, H, N]   the WKV outputs
 *   r, k, v, g      : x_dtype [n_rows, H, N] (x_dtype WKV7_F32 or WKV7_BF16)
 *   r_k, ln_w, ln_b : fp32 [H, N]
 *   eps             : finite, >= 0
 *   y               : fp32 [n_rows, H, N]; may be the same pointer as o (in
 *                     place), otherwise it overlaps no argument
 */
WKV7_API wkv7_status wkv7_tmix_tail(int n_rows, int H, int N, wkv7_dtype x_dtype,
                      const float *o, const void *r, const void *k, const void *v,
                      const void *g, const float *r_k, const float *ln_w,
                      const float *ln_b, float eps, float *y, cudaStream_t stream);

/*
 * wkv7_verify -- the recurrence over T = K + 1 tokens per row from a read-only
 * state, keeping every position's state: the WKV part of one speculative step
 * of the RWKV-Infer-Next page ("Inference. One speculative step": the base
 * model processes [t, d1 .. dK] in one forward, the sampler accepts the drafts
 * up to the first mismatch, the recurrent state is rolled back to the accepted
 * prefix).  For each row b, head h and position t = 0 .. T-1:
 *     S_{-1} = state[b, h] ;  S_t = step(S_{t-1}, x[b, t, h]) ;  o[b, t, h] = S_t^T r[b, t, h]
 *
 *   T                  : 1 .. 8 tokens per row (K = T - 1 drafts)
 *   r, w, k, v, kk, a  : fp32 [B, T, H, N]
 *   state              : fp32 [B, H, N, N]     read only
 *   o                  : fp32 [B, T, H, N]
 *   states             : fp32 [T, B, H, N, N]  states[t] = S_t of every (row, head):
 *                        states[t] has the layout of `state`, so a batch that
 *                        accepts the same length everywhere can use it as is
 * o and states overlap no input and not each other (WKV7_ERR_INVALID_ARG).
 *
 * wkv7_verify_commit -- the rollback: state[b] = states[accept_len[b] - 1][b]
 * for every head, or unchanged when accept_len[b] = 0.  accept_len is a DEVICE
 * int32 [B] (written by the sampler, so no host round trip is needed); a value
 * outside 0 .. T leaves that row unchanged and is reported by
 * wkv7_check_device_status (WKV7_ERR_DEVICE_BOUNDS).  The pages have no
 * separate rollback call; it completes wkv7_verify's per-position states.
 */
WKV7_API wkv7_status wkv7_verify(int B, int T, int H, int N,
                      const float *r, const float *w, const float *k,
                      const float *v, const float *kk, const float *a,
                      const float *state, float *o, float *states, cudaStream_t stream);
WKV7_API wkv7_status wkv7_verify_commit(int B, int T, int H, int N, const float *states,
                      const int32_t *accept_len, float *state, cudaStream_t stream);

/*
 * wkv7_prefill_workspace_size -- bytes of device workspace with which
 * wkv7_prefill can use every schedule for this shape (may be 0; the result
 * depends only on the arguments).  It holds:
 *   - the longest-first order of the sequences, 4 bytes per sequence rounded
 *     up to 256, for 2 <= num_seqs <= 4096 (required: a smaller workspace
 *     returns WKV7_ERR_WORKSPACE);
 *   - for T_total >= 1024, scratch for the tail split (optional): 512 state
 *     slots of 16 KB, then 256 bytes per token-head for up to
 *     min(T_total * H, 2^20) token-heads.  When the (sequence, head)
 *     pairs do not fill the last wave of CTAs (0 < P mod SMs <= SMs / 2, at
 *     most 80 pairs), the pairs of that wave are cut into chunk-aligned
 *     segments that run concurrently; a segment after the first runs from a
 *     zero state and once more from the identity state with v = 0, and two
 *     small kernels chain the true boundary states and add the carried-in
 *     state's contribution to the outputs (exact up to rounding: the
 *     recurrence is linear in the state).  This needs cu_seqlens_host; with
 *     less scratch than a plan needs, or without the host copy, every pair
 *     runs whole.
 */
WKV7_API size_t wkv7_prefill_workspace_size(int num_seqs, int T_total, int H, int N);

/*
 * wkv7_prefill -- the recurrence over packed variable-length sequences.
 *
 * The parallel "prefill(ids, state:)" pass of the SwiftRWKV inference page
 * (a whole prompt in one launch, "What the prefill path is made of"), with
 * the batch packed by cu_seqlens instead of right padding.  The result equals
 * running wkv7_step over each sequence's tokens in order.
 *
 *   num_seqs        : number of sequences (>= 0)
 *   T_total         : total tokens (>= 0)
 *   cu_seqlens      : DEVICE int32 [num_seqs + 1]; sequence b owns tokens
 *                     cu_seqlens[b] .. cu_seqlens[b+1]-1; cu_seqlens[0] = 0,
 *                     non-decreasing, cu_seqlens[num_seqs] = T_total.
 *                     Zero-length sequences are allowed.
 *   cu_seqlens_host : optional HOST copy of the same array (NULL allowed).
 *                     When given it is validated on the host and used to
 *                     schedule long sequences first and to plan the tail
 *                     split; it must equal the device array.  When NULL the
 *                     device validates cu_seqlens and a malformed array is
 *                     reported by wkv7_check_device_status.
 *   x_dtype         : the type of r, k, v, kk, a, and the kernel that runs:
 *                     WKV7_BF16 -- bf16, the chunked tensor-core kernel (the
 *                       WY/UT form, contractions at tf32 with fp32 accumulation);
 *                     WKV7_TF32 -- fp32 inputs through the same chunked kernel
 *                       (read at full precision, contracted at tf32: the same
 *                       error bound and domain as bf16 inputs);
 *                     WKV7_F32 -- fp32 inputs through an exact token-serial
 *                       kernel (fp32 arithmetic throughout, no domain limit)
 *   r, k, v, kk, a  : x_dtype [T_total, H, N]  (token-major)
 *   w               : fp32 [T_total, H, N]     log-decay
 *   initial_state   : fp32 [num_seqs, H, N, N] or NULL (= zeros)
 *   final_state     : fp32 [num_seqs, H, N, N] or NULL (not written); may be
 *                     the same pointer as initial_state (in-place carry), but
 *                     must not partially overlap it
 *   o               : fp32 [T_total, H, N]     outputs of every token
 *   workspace       : device memory, 16-byte aligned, of workspace_bytes
 *                     bytes: wkv7_prefill_workspace_size(...) for every
 *                     schedule, at least its sequence-order part (may be NULL
 *                     when that part is 0).  Its contents need not be
 *                     initialised and are not preserved; it must not overlap
 *                     any other argument.  Calls that overlap on the GPU must
 *                     use distinct workspaces.
 *
 * Domain of the chunked formulation (WKV7_BF16, WKV7_TF32): w >= -1 elementwise
 * (every RWKV-7 model has w in (-0.6066, 0)).  The chunked kernel takes a
 * chunk's decay factors relative to its 32nd token, so each scaled operand
 * carries a factor within e^{+-32} and the chunk's removal block, where one
 * channel's growing factor meets another's through the UT transform, within
 * e^{64}: finite in fp32 with a wide margin.  (At w = -2.5 on some channels
 * and 0 on others that block overflows.)  The kernel checks the domain on the
 * device: a w below -1 (or -inf) is reported by wkv7_check_device_status as
 * WKV7_ERR_INVALID_ARG, and the outputs of that call are then unspecified
 * (they may hold inf or NaN).  WKV7_F32 inputs take the token-serial kernel,
 * which has no such limit.
 */
WKV7_API wkv7_status wkv7_prefill(int num_seqs, int T_total, int H, int N,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                         wkv7_dtype x_dtype,
                         const void *r, const float *w, const void *k,
                         const void *v, const void *kk, const void *a,
                         const float *initial_state, float *final_state, float *o,
                         void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * wkv7_step_cast, wkv7_prefill_cast -- wkv7_step and wkv7_prefill with the output
 * o in o_dtype: WKV7_F32, or WKV7_BF16 (each element of the fp32 result rounded
 * to nearest even; o then holds 2 bytes per element and all its bounds and
 * overlap rules use that size).  The SwiftRWKV inference page converts the WKV
 * output to the model's compute type as soon as the recurrence has produced
 * it, while the recurrent state itself stays fp32 (its
 * castWKVOutputToComputeDType switch); the state stays fp32 here too.
 * With a bf16 output the tail split keeps its partial outputs in fp32
 * scratch rows and rounds once, after the correction (it then needs twice
 * the readout scratch; with less, every pair runs whole).
 */
WKV7_API wkv7_status wkv7_step_cast(int B, int H, int N,
                      const float *r, const float *w, const float *k,
                      const float *v, const float *kk, const float *a,
                      float *state, void *o, wkv7_dtype o_dtype, cudaStream_t stream);
WKV7_API wkv7_status wkv7_prefill_cast(int num_seqs, int T_total, int H, int N,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                         wkv7_dtype x_dtype,
                         const void *r, const float *w, const void *k,
                         const void *v, const void *kk, const void *a,
                         const float *initial_state, float *final_state, void *o,
                         wkv7_dtype o_dtype, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * wkv7_prefill_state -- wkv7_prefill_cast with initial_state and final_state
 * in state_dtype: WKV7_F32, WKV7_F16 or WKV7_BF16 (both the same type).  A
 * 16-bit initial state is widened to fp32 exactly, the whole prefill runs with
 * the fp32 state of wkv7_prefill, and the final state is rounded to nearest
 * even once, when it is stored.  The counterpart of wkv7_step_state for the
 * prompt that fills a 16-bit state cache; all other rules as wkv7_prefill_cast,
 * with the byte sizes of the chosen state type.
 */
WKV7_API wkv7_status wkv7_prefill_state(int num_seqs, int T_total, int H, int N,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                         wkv7_dtype x_dtype,
                         const void *r, const float *w, const void *k,
                         const void *v, const void *kk, const void *a,
                         const void *initial_state, void *final_state, wkv7_dtype state_dtype,
                         void *o, wkv7_dtype o_dtype, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * wkv7_prefill_padded -- wkv7_prefill_cast over a right-padded batch: row b of
 * the [B, T_max, H, N] inputs holds lens[b] real tokens followed by padding.
 * The SwiftRWKV inference page feeds its batched prefill this way (right
 * padding, each row ending on its last real token).  The result for row b is
 * that of a packed sequence of its lens[b] tokens; positions past lens[b] of o
 * are not written.
 *
 *   lens      : DEVICE int32 [B], 0 <= lens[b] <= T_max (a value outside is
 *               reported by wkv7_check_device_status and that row is skipped)
 *   lens_host : optional HOST copy of lens (validated; used for scheduling)
 *   r, k, v, kk, a : x_dtype [B, T_max, H, N];  w : fp32 [B, T_max, H, N]
 *   o         : o_dtype [B, T_max, H, N]
 *   initial_state, final_state : fp32 [B, H, N, N], as wkv7_prefill
 *   workspace : as wkv7_prefill with num_seqs = B, T_total = B * T_max
 */
WKV7_API wkv7_status wkv7_prefill_padded(int B, int T_max, int H, int N,
                         const int32_t *lens, const int32_t *lens_host,
                         wkv7_dtype x_dtype,
                         const void *r, const float *w, const void *k,
                         const void *v, const void *kk, const void *a,
                         const float *initial_state, float *final_state, void *o,
                         wkv7_dtype o_dtype, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * wkv7_prefill_noalloc -- wkv7_prefill without a caller-supplied workspace.
 *
 * For callers that cannot allocate device memory when they run the prefill:
 * a serving engine whose memory plan reserves the whole device up front so
 * that request handling never allocates, code recorded during CUDA stream
 * capture (where cudaMalloc is not permitted), or a host program that only
 * receives pointers to buffers owned by someone else.  The pages have no
 * counterpart; the arguments are those of wkv7_prefill without `workspace`.
 *
 * The scratch this call needs (the longest-first order of the sequences)
 * lives in a fixed device array of WKV7_NOALLOC_MAX_SEQS int32 entries
 * (16 KB) that the library reserves on every GPU that loads it, until the
 * process exits.  num_seqs > WKV7_NOALLOC_MAX_SEQS returns
 * WKV7_ERR_WORKSPACE.  The call allocates nothing.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current); make that first call before any stream capture.
 * All calls on a device share the array: calls that overlap on the GPU (on
 * different streams, or launched from different threads without ordering)
 * race on it and must be serialised by the caller.  Each call overwrites the
 * entries it uses before reading them.
 */
#define WKV7_NOALLOC_MAX_SEQS 4096

WKV7_API wkv7_status wkv7_prefill_noalloc(int num_seqs, int T_total, int H, int N,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                         wkv7_dtype x_dtype,
                         const void *r, const float *w, const void *k,
                         const void *v, const void *kk, const void *a,
                         const float *initial_state, float *final_state, float *o,
                         cudaStream_t stream);

/*
 * wkv7_prefill_backward -- gradients of a wkv7_prefill call, for training.
 *
 * The Pantheon RWKV-X page lists training (a forward with callbacks) among the
 * Foundry engine's features, and the SwiftRWKV inference page notes that a
 * fused kernel is opaque to autograd; this call is the written-out derivative
 * of the recurrence of wkv7_step (Core AI model zoo, section 1) for the loss
 *     L = sum_t <d_o_t, o_t> + sum_b <d_final_state_b, S_final_b>,
 * i.e. the vector-Jacobian product of (o, final_state) with (d_o,
 * d_final_state).  It recomputes the states itself from the inputs: it needs no
 * saved forward activations beyond the inputs of the wkv7_prefill call.
 *
 *   num_seqs .. a    : exactly the arguments of the wkv7_prefill call being
 *                      differentiated (same layouts, dtypes and sequence
 *                      rules; cu_seqlens_host optional and validated;
 *                      WKV7_TF32 and WKV7_F32 both mean fp32 inputs here)
 *   initial_state    : fp32 [num_seqs, H, N, N] or NULL (= zeros), as given
 *                      to wkv7_prefill
 *   d_o              : fp32 [T_total, H, N]     gradient of the loss w.r.t. o
 *   d_final_state    : fp32 [num_seqs, H, N, N] or NULL (= zeros)
 *   dr, dw, dk, dv, dkk, da : fp32 [T_total, H, N]  (written; dw is the
 *                      gradient w.r.t. the log-decay w)
 *   d_initial_state  : fp32 [num_seqs, H, N, N] or NULL (not written)
 *   workspace        : device memory, 16-byte aligned, of at least
 *                      wkv7_prefill_backward_workspace_size(num_seqs, T_total,
 *                      H, N) bytes (about 1.5 KB per token and head: the
 *                      state at every 64-token boundary plus five 64 x 64
 *                      matrices per chunk); contents need not be initialised.
 *
 * Every written range must not overlap any other argument.  Zero-length
 * sequences give d_initial_state = d_final_state.  Same domain as the chunked
 * wkv7_prefill (w >= -1, for either input type), checked on the device the
 * same way: a w below it is reported by wkv7_check_device_status as
 * WKV7_ERR_INVALID_ARG.  Stream-ordered, no synchronisation; a malformed
 * device cu_seqlens (when no host copy is given) is reported by
 * wkv7_check_device_status and leaves the token gradients unwritten.
 */
WKV7_API size_t wkv7_prefill_backward_workspace_size(int num_seqs, int T_total, int H, int N);
WKV7_API wkv7_status wkv7_prefill_backward(int num_seqs, int T_total, int H, int N,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                         wkv7_dtype x_dtype,
                         const void *r, const float *w, const void *k,
                         const void *v, const void *kk, const void *a,
                         const float *initial_state, const float *d_o, const float *d_final_state,
                         float *dr, float *dw, float *dk, float *dv, float *dkk, float *da,
                         float *d_initial_state, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * wkv7_diag_bounded_wait -- a diagnostic of the timeout path.  Launches one
 * device-side wait on a barrier that nothing completes, through the same
 * bounded wait (global-timer limit plus a poll count) and status report the
 * kernels use for every mbarrier wait.  After timeout_us (1 .. 2,000,000) the
 * device gives up and sets the timeout bit of the status word, exactly as an
 * expired wait inside a kernel would; wkv7_check_device_status then returns
 * WKV7_ERR_TIMEOUT (and clears it) and the context stays usable.  No fault and
 * no hang: the wait always ends.  Stream-ordered; returns WKV7_ERR_INVALID_ARG
 * for a timeout outside the range, WKV7_ERR_CUDA if the launch fails.
 */
WKV7_API wkv7_status wkv7_diag_bounded_wait(unsigned timeout_us, cudaStream_t stream);

/* Static English text for a status code (never NULL). */
WKV7_API const char *wkv7_status_string(wkv7_status status);

/*
 * wkv7_check_device_status -- synchronise `stream`, then read and clear the
 * current device's status word.  Returns WKV7_OK, WKV7_ERR_TIMEOUT,
 * WKV7_ERR_DEVICE_BOUNDS, WKV7_ERR_INVALID_ARG (malformed device cu_seqlens,
 * or a w below the chunked kernels' domain) or WKV7_ERR_CUDA (the
 * synchronisation itself failed).
 *
 * The library looks up the device address of this status word (and of the
 * fixed scratch of wkv7_prefill_noalloc) once per device and keeps it for the
 * life of the process.  After cudaDeviceReset, or any other teardown of a
 * device's primary context, those cached addresses are stale: do not call the
 * library on that device again in the same process.
 */
WKV7_API wkv7_status wkv7_check_device_status(cudaStream_t stream);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
WKV7_API const char *wkv7_last_cuda_error(void);

/* ABI version: 100 * major + minor. */
WKV7_API int wkv7_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WKV7_H */
