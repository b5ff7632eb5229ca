/*
 * kda.h - C ABI of the KDA (Kimi Delta Attention) library for GB300 (sm_103a).
 *
 * The method is the per-channel gated delta rule of the web page
 * "研究KimiK3，我发现大模型正在学会“管理自己的计算”" (pwwt.cn/news/3763336),
 * called "the K3 essay" below. Per sequence and head, for t = 1..T:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T   (§四)
 *     o_t = S_t^T q_t                                                         (§二.1)
 *
 * with S a d_k x d_v float32 state, alpha_t in [0,1]^{d_k} a per-channel gate
 * and beta_t a scalar write strength. Prefill evaluates it chunk by chunk in
 * the WY form of §六 (chunks of 64 tokens: state passed between chunks, the
 * tokens inside a chunk handled as a few dense products); decode applies one
 * token in place.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers, row-major and contiguous, 16-byte
 *    aligned (kda_prefill_host and kda_prefill_fp8_host alone take host
 *    buffers). The caller owns every buffer; the library allocates nothing,
 *    never synchronises the stream, and launches all its work on `stream`
 *    (the two host-buffer calls also use two copy streams of their own, and
 *    kda_prefill_segmented three streams of its own, all joined back into
 *    `stream`).
 *  - Layouts: q, k, alpha [.., T, H, d_k]; v, o [.., T, H, d_v]; beta [.., T, H];
 *    states [N, H, d_k, d_v] with d_v fastest. alpha and beta are float32;
 *    q, k, v and o share `qkv_dtype`; states are float32.
 *  - Supported: d_k, d_v in {64, 128}. Other sizes return KDA_ERR_UNSUPPORTED.
 *  - Gates: alpha is used as given (linear, not log); alpha = 0 is allowed and
 *    erases the channel. beta may be any finite value.
 *  - Errors: argument checks run before any launch and return a status with
 *    nothing launched; the message is in kda_last_error() (per thread).
 *    A failed launch returns KDA_ERR_CUDA. Device-side checks never trap: they
 *    write a code to a caller-visible status word and skip the work.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer   */
    KDA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d_k = 96)   */
    KDA_ERR_CUDA = 3,          /* a CUDA call or launch failed                */
    KDA_ERR_DEVICE_CHECK = 4,  /* a device-side check failed (status word)    */
    KDA_ERR_WORKSPACE = 5      /* workspace missing or too small              */
} kda_status_t;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype_t;

/* Prefill implementation choice (kda_prefill picks KDA_ALGO_AUTO). */
typedef enum {
    KDA_ALGO_AUTO = 0,  /* tensor-core path for bf16 d=128, SIMT otherwise       */
    KDA_ALGO_SIMT = 1,  /* fp32 CUDA-core chunk kernel (any supported dtype/d)   */
    KDA_ALGO_TC = 2     /* tcgen05/TMEM chunk kernel: bf16, d_k = d_v = 128 only */
} kda_algo_t;

/*
 * Gate kinds (the entry points ending in _gate / _slots take one). The K3
 * essay's §四 places KDA's per-channel gate next to the scalar gate of Gated
 * DeltaNet; with no gate the update is the plain delta rule of §三.
 *   KDA_GATE_CHANNEL  alpha [.., H, d_k]: one gate per key channel (KDA)
 *   KDA_GATE_SCALAR   alpha [.., H]: one gate per token and head, the same for
 *                     every channel (Gated DeltaNet); 4-byte aligned suffices
 *   KDA_GATE_NONE     alpha is not read and may be NULL: alpha = 1 (DeltaNet)
 * Each kind computes exactly what KDA_GATE_CHANNEL computes with alpha
 * broadcast over the channels (all ones for NONE).
 */
typedef enum { KDA_GATE_CHANNEL = 0, KDA_GATE_SCALAR = 1, KDA_GATE_NONE = 2 } kda_gate_t;

/* Device-side status codes written to `device_status`. */
#define KDA_DEV_OK 0
#define KDA_DEV_BAD_CU_SEQLENS 1   /* cu[0] != 0, decreasing, or cu[N] != T_total */
#define KDA_DEV_BAD_SLOT 2         /* a state slot outside [0, pool_size)          */

/*
 * kda_prefill - chunkwise prefill of B equal-length sequences (K3 essay §四
 * update, evaluated with §六's chunking and WY form).
 *
 *   q, k         [B, T, H, d_k]  qkv_dtype          (read)
 *   v            [B, T, H, d_v]  qkv_dtype          (read)
 *   alpha        [B, T, H, d_k]  float32, in [0,1]  (read)
 *   beta         [B, T, H]       float32            (read)
 *   initial_state[B, H, d_k, d_v] float32 or NULL (zeros)            (read)
 *   o            [B, T, H, d_v]  qkv_dtype: o_t = S_t^T q_t          (written)
 *   final_state  [B, H, d_k, d_v] float32 or NULL (not written)      (written)
 *
 * final_state may equal initial_state (updated in place). T = 0 copies the
 * initial state (or zeros) to final_state. Returns KDA_OK once the work is
 * queued on `stream`.
 */
kda_status_t kda_prefill(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                         const float *alpha, const float *beta, const float *initial_state,
                         void *o, float *final_state, int B, int T, int H, int d_k, int d_v,
                         kda_stream_t stream);

/* kda_prefill with an explicit implementation choice (KDA_ALGO_TC on an
 * unsupported dtype or size returns KDA_ERR_UNSUPPORTED). */
kda_status_t kda_prefill_ex(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                            const float *alpha, const float *beta, const float *initial_state,
                            void *o, float *final_state, int B, int T, int H, int d_k, int d_v,
                            kda_algo_t algo, kda_stream_t stream);

/*
 * kda_varlen_prefill - prefill of N sequences packed along the token axis.
 * Sequence n owns tokens cu_seqlens[n] .. cu_seqlens[n+1]-1 and runs its own
 * recurrence from its own initial state, with its own chunk grid starting at
 * its first token; results are bitwise equal to kda_prefill on that sequence
 * alone.
 *
 *   q, k, alpha  [T_total, H, d_k];  v, o [T_total, H, d_v];  beta [T_total, H]
 *   cu_seqlens   [N + 1] int32, DEVICE memory; must start at 0, never decrease
 *                and end at T_total (checked on the device).
 *   initial_state / final_state  [N, H, d_k, d_v] float32, nullable as above.
 *   workspace    device scratch of at least kda_varlen_workspace_bytes(N, H,
 *                d_k, d_v) bytes, 256-byte aligned; its contents on entry do
 *                not matter. Calls sharing a workspace must not overlap.
 *   device_status DEVICE int32 or NULL: set to KDA_DEV_OK or a KDA_DEV_* code
 *                when the call's kernels run; on a code, no o or state is
 *                written by this call.
 */
kda_status_t kda_varlen_prefill(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                const float *alpha, const float *beta,
                                const float *initial_state, void *o, float *final_state,
                                const int32_t *cu_seqlens, int N, int T_total, int H, int d_k,
                                int d_v, void *workspace, size_t workspace_bytes,
                                int32_t *device_status, kda_stream_t stream);

/* Workspace bytes kda_prefill, kda_prefill_ex, kda_prefill_gate and
 * kda_prefill_fp8 need: always 0. Equal-length sequences need no scratch (the
 * state of every chunk stays on chip), so those calls take no workspace
 * argument; the function exists so that callers that size workspaces
 * generically can treat every prefill alike. */
size_t kda_prefill_workspace_bytes(int B, int T, int H, int d_k, int d_v);

/* Workspace bytes kda_varlen_prefill needs for N sequences (0 < result). */
size_t kda_varlen_workspace_bytes(int N, int H, int d_k, int d_v);

/*
 * kda_prefill_segmented - kda_prefill of ONE long sequence (B = 1) with its
 * token axis cut into segments that run at the same time, for sequences far
 * longer than the batch is wide (few heads leave most of the GPU idle while
 * each head walks its chunks in order).
 *
 * The update is an affine map of the state, S_t = A_t S_{t-1} + B_t (K3
 * essay §六), with the transition from token j to t the product A_t..A_{j+1}
 * (§五). Over a segment, S_end = Phi S_start + b. Segment 0 runs from
 * initial_state; each later segment runs once from zero (its outputs and b)
 * and once with v = 0 from the identity (its outputs z_t = Phi_t^T q_t and
 * Phi), all at once; then S_start of every segment follows in float32 and
 * o_t += S_start^T z_t corrects the later segments' outputs (bf16 operands,
 * float32 accumulation). Every segment boundary is a multiple of 64 tokens.
 *
 *   q, k, v, alpha, gate, beta, initial_state, o, final_state: as
 *                kda_prefill_gate with B = 1 (final_state may equal
 *                initial_state).
 *   segments     0: the library's plan (no split when it would not pay, e.g.
 *                more than 38 heads, or a short sequence); 1: no split (a
 *                plain kda_prefill); 2..4096: that many segments (fewer when
 *                the sequence has too few chunks; H <= 65535).
 *   workspace    device scratch of kda_prefill_segmented_workspace_bytes(...)
 *                bytes (0 when there is no split; then it may be NULL),
 *                256-byte aligned; contents on entry do not matter. About
 *                0.5 KB per token-head of the later segments. Calls sharing a
 *                workspace must not overlap.
 * Results agree with kda_prefill within the bf16 tolerance of the tensor-core
 * path; they are not bitwise equal to it (the later segments' outputs are
 * rounded to bf16 once before the correction and once after).
 * A split needs bf16 q/k/v and d_k = d_v = 128 (KDA_ERR_UNSUPPORTED for
 * segments >= 2 otherwise; segments = 0 then runs kda_prefill). Streams: the
 * segments run on three streams of the library's own (created once per
 * device), forked from and joined back into `stream`; the call can be
 * captured into a CUDA graph (make the first split call on a device before
 * any capture: it creates those streams). Errors: argument, alignment and workspace
 * checks return before any launch (KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED,
 * KDA_ERR_WORKSPACE); if a launch fails midway, `stream` still waits for
 * everything already queued and the call returns KDA_ERR_CUDA. Calls from
 * several host threads on one device are serialised while they queue work.
 */
kda_status_t kda_prefill_segmented(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                   const float *alpha, kda_gate_t gate, const float *beta,
                                   const float *initial_state, void *o, float *final_state, int B, int T, int H,
                                   int d_k, int d_v, int segments, void *workspace, size_t workspace_bytes,
                                   kda_stream_t stream);

/* Workspace bytes of kda_prefill_segmented for these arguments. */
size_t kda_prefill_segmented_workspace_bytes(int B, int T, int H, int d_k, int d_v, kda_dtype_t qkv_dtype,
                                             int segments);

/* The split kda_prefill_segmented makes for these arguments: the number of
 * segments, the tokens of segment 0 and of each later segment (the last one
 * ends at T). No split: *n_segments = 1, *first_tokens = T. */
kda_status_t kda_prefill_segment_plan(int B, int T, int H, int d_k, int d_v, kda_dtype_t qkv_dtype, int segments,
                                      int *n_segments, int *first_tokens, int *segment_tokens);

/*
 * kda_varlen_prefill_noalloc - kda_varlen_prefill without a workspace, for
 * callers that must not allocate device memory (engines whose device memory
 * is planned up front and may not grow on the request path, plug-ins that
 * are handed only the call's tensors, paths where an allocation would
 * synchronise). The method has no counterpart: this is an interface choice.
 *
 * Arguments, layouts and results are those of kda_varlen_prefill. The small
 * scratch it needs (sequence order, work counter, status word) is a fixed
 * array inside the library, present on every GPU that loads the library
 * until the process exits; it holds at most KDA_NOALLOC_MAX_SEQS sequences,
 * and larger N is rejected with KDA_ERR_UNSUPPORTED before anything runs.
 * The first call on a device looks up that array's device address once
 * (with the device current); make this first call before any stream capture.
 * The address is kept until the process exits, so do not use this entry
 * point on a device after cudaDeviceReset.
 * All calls share the one array and each call rewrites what it uses, so calls
 * that overlap on the GPU (different streams, or different host threads on
 * the same device) race and must be serialised by the caller.
 */
#define KDA_NOALLOC_MAX_SEQS 16384
kda_status_t kda_varlen_prefill_noalloc(const void *q, const void *k, const void *v,
                                        kda_dtype_t qkv_dtype, const float *alpha, const float *beta,
                                        const float *initial_state, void *o, float *final_state,
                                        const int32_t *cu_seqlens, int N, int T_total, int H, int d_k,
                                        int d_v, int32_t *device_status, kda_stream_t stream);

/*
 * kda_prefill_host - kda_prefill_gate on HOST buffers: q, k, v, alpha, beta,
 * initial_state (nullable), o and final_state (nullable) are host pointers in
 * the layouts of kda_prefill_gate (no alignment needed); `workspace` is device
 * memory of at least kda_prefill_host_workspace_bytes(...) bytes, 16-byte
 * aligned, owned by the caller.
 *
 * The tokens go to the device in pieces of `piece_tokens` tokens along T (0:
 * the library picks about 32 MiB of input per piece; otherwise a positive
 * multiple of 64), each piece is one kda_prefill_gate launch on `stream` that
 * continues from the state the previous piece left in the workspace (the
 * chunk-to-chunk state passing of the K3 essay §六.1), and each piece's o
 * returns while later pieces are still in flight. The result is bit for bit
 * that of kda_prefill_gate run piece by piece on the device with the state
 * passed between the pieces; against one kda_prefill_gate call over all T
 * tokens it differs only by rounding at the piece boundaries (one piece, i.e.
 * piece_tokens >= T, gives the bits of the single call).
 *
 * Ordering: everything is queued after the work already on `stream`, and work
 * queued on `stream` afterwards starts once o and final_state are in host
 * memory; synchronise `stream` before reading them. The call returns once all
 * copies are queued. With pageable host memory the driver copies
 * synchronously, so the call returns only after those copies, and nothing
 * overlaps; the result is the same. Page-locked host memory gives the
 * overlap. The first call on a device
 * creates two copy streams and a few events that live until the process
 * exits; calls are serialised by a lock while they queue their work.
 *
 * Errors: as kda_prefill_gate; a device pointer where a host buffer is
 * expected returns KDA_ERR_INVALID_ARG, a missing or short workspace
 * KDA_ERR_WORKSPACE, both before anything is queued.
 */
kda_status_t kda_prefill_host(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                              const float *alpha, kda_gate_t gate, const float *beta,
                              const float *initial_state, void *o, float *final_state, int B, int T,
                              int H, int d_k, int d_v, kda_algo_t algo, int piece_tokens, void *workspace,
                              size_t workspace_bytes, kda_stream_t stream);

/* Device workspace bytes kda_prefill_host needs for these sizes (0 for invalid
 * arguments): three piece buffers of every tensor and one set of states. */
size_t kda_prefill_host_workspace_bytes(int B, int T, int H, int d_k, int d_v, kda_dtype_t qkv_dtype,
                                        kda_gate_t gate, int piece_tokens);

/*
 * kda_prefill_fp8_host - kda_prefill_fp8 on HOST buffers, through the piece
 * pipeline of kda_prefill_host: q, k, v (E4M3 codes), q_scale, k_scale,
 * v_scale (E8M0), alpha, beta, initial_state (nullable), o (bf16) and
 * final_state (nullable) are host pointers in the layouts of kda_prefill_fp8;
 * `workspace` is device memory of at least kda_prefill_fp8_host_workspace_bytes
 * bytes, 16-byte aligned. The host link carries 1 byte per q, k, v element
 * instead of 2, which is where the FP8 format pays off: the end-to-end call is
 * bound by that link. Result, ordering, piece size and errors as for
 * kda_prefill_host (bit for bit kda_prefill_fp8 run piece by piece on the
 * device with the state passed between the pieces). d_k = d_v = 128 only.
 */
kda_status_t kda_prefill_fp8_host(const uint8_t *q, const uint8_t *k, const uint8_t *v, const uint8_t *q_scale,
                                  const uint8_t *k_scale, const uint8_t *v_scale, const float *alpha,
                                  kda_gate_t gate, const float *beta, const float *initial_state, void *o,
                                  float *final_state, int B, int T, int H, int d_k, int d_v, int piece_tokens,
                                  void *workspace, size_t workspace_bytes, kda_stream_t stream);

/* Device workspace bytes kda_prefill_fp8_host needs (0 for invalid arguments). */
size_t kda_prefill_fp8_host_workspace_bytes(int B, int T, int H, int d_k, int d_v, kda_gate_t gate,
                                            int piece_tokens);

/*
 * kda_decode_step - one recurrent step per (sequence, head), in place
 * (K3 essay §四 update for a single token, §二.1 read-out):
 *     S' = Diag(alpha) S;  e = beta (v - S'^T k);  S <- S' + k e^T;  o = S^T q
 *
 *   q, k   [N, H, d_k] qkv_dtype;  v, o [N, H, d_v] qkv_dtype
 *   alpha  [N, H, d_k] float32;    beta [N, H] float32
 *   state  [N, H, d_k, d_v] float32, read and overwritten in place
 */
kda_status_t kda_decode_step(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                             const float *alpha, const float *beta, float *state, void *o,
                             int N, int H, int d_k, int d_v, kda_stream_t stream);

/*
 * kda_prefill_gate - kda_prefill_ex with a gate kind (see kda_gate_t): alpha is
 * [B, T, H, d_k] (CHANNEL), [B, T, H] (SCALAR) or unused (NONE). Everything
 * else as kda_prefill_ex.
 */
kda_status_t kda_prefill_gate(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                              const float *alpha, kda_gate_t gate, const float *beta,
                              const float *initial_state, void *o, float *final_state, int B, int T,
                              int H, int d_k, int d_v, kda_algo_t algo, kda_stream_t stream);

/*
 * kda_prefill_fp8 - kda_prefill_gate on FP8 inputs in the MX block format:
 * q, k, v hold FP8 E4M3 codes and every 32 consecutive channels (values) of a
 * token-head share one E8M0 scale byte t, the power of two 2^(t - 127):
 *
 *   q, k        [B, T, H, d_k] uint8 (E4M3)      q_scale, k_scale [B, T, H, d_k/32] uint8
 *   v           [B, T, H, d_v] uint8 (E4M3)      v_scale          [B, T, H, d_v/32] uint8
 *   o           [B, T, H, d_v] bfloat16 (written)
 *
 * The result is that of kda_prefill_gate with bf16 q, k, v holding the
 * dequantised values (code x 2^(t-127), exactly representable in bf16 for
 * t in [1, 254]); the inputs simply take half the bytes. Tensor-core kernel
 * only: d_k = d_v = 128. Scale bytes 0 and 255 are not supported (their
 * values are undefined); E4M3 NaN codes propagate.
 */
kda_status_t kda_prefill_fp8(const uint8_t *q, const uint8_t *k, const uint8_t *v, const uint8_t *q_scale,
                             const uint8_t *k_scale, const uint8_t *v_scale, const float *alpha,
                             kda_gate_t gate, const float *beta, const float *initial_state, void *o,
                             float *final_state, int B, int T, int H, int d_k, int d_v, kda_stream_t stream);

/*
 * State slots for serving: a pool of recurrent states that outlives the calls
 * (prefill, then any number of decode steps, or a long prompt prefilled in
 * pieces), each request owning one slot. Both calls below read a sequence's
 * state from its slot and write the new state back into the same slot.
 *
 *   state_pool  [pool_size, H, d_k, d_v] float32, DEVICE, read and written
 *   slots       [N] int32, DEVICE: sequence n uses slot s = slots[n]; a value
 *               -1 - s means "slot s, starting from the zero state" (a new
 *               request). Two sequences of one call must not share a slot.
 *   device_status  DEVICE int32 or NULL: set to KDA_DEV_OK, or to
 *               KDA_DEV_BAD_SLOT when a slot lies outside [0, pool_size) (and
 *               KDA_DEV_BAD_CU_SEQLENS as for kda_varlen_prefill).
 *
 * Prefilling a prompt in pieces, each piece continuing from the slot's state,
 * gives the result of one prefill of the whole prompt (to rounding), because
 * the state carries everything the recurrence knows (§六.1).
 */

/*
 * kda_varlen_prefill_slots - kda_varlen_prefill whose initial and final states
 * live in `state_pool` at `slots`, with a gate kind. On KDA_DEV_BAD_CU_SEQLENS
 * or KDA_DEV_BAD_SLOT nothing is written (no o, no state). The workspace is
 * the one of kda_varlen_prefill (kda_varlen_workspace_bytes).
 */
kda_status_t kda_varlen_prefill_slots(const void *q, const void *k, const void *v,
                                      kda_dtype_t qkv_dtype, const float *alpha, kda_gate_t gate,
                                      const float *beta, float *state_pool, const int32_t *slots,
                                      int pool_size, void *o, const int32_t *cu_seqlens, int N,
                                      int T_total, int H, int d_k, int d_v, void *workspace,
                                      size_t workspace_bytes, int32_t *device_status,
                                      kda_stream_t stream);

/*
 * kda_decode_step_slots - kda_decode_step on the states state_pool[slots[n]]
 * (updated in place), with a gate kind: alpha [N, H, d_k] (CHANNEL), [N, H]
 * (SCALAR) or unused (NONE). A sequence whose slot is out of range is skipped
 * (its o is not written) and sets KDA_DEV_BAD_SLOT in `device_status`; the
 * others run.
 */
kda_status_t kda_decode_step_slots(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                   const float *alpha, kda_gate_t gate, const float *beta,
                                   float *state_pool, const int32_t *slots, int pool_size, void *o,
                                   int N, int H, int d_k, int d_v, int32_t *device_status,
                                   kda_stream_t stream);

/*
 * kda_device_errors - diagnostic: reads the library's device-side error word
 * (0 = none). A nonzero value means a kernel stopped early because one of its
 * bounded waits ran out (its outputs are then invalid); the kernel returned
 * instead of hanging. Synchronises with the device (a blocking copy of one
 * int). reset != 0 clears the word after reading.
 */
kda_status_t kda_device_errors(int *errors, int reset);

/*
 * kda_prefill_backward - gradients of the prefill (training). The pages give
 * no gradients; they follow from the chain rule applied to the K3 essay's
 * §四 update and §二.1 read-out, evaluated with §六's chunks in reverse. For
 * L = sum_t <d_o_t, o_t> + <d_final_state, S_T> it returns dL/dq, dL/dk,
 * dL/dv, dL/dalpha, dL/dbeta and dL/dS_0 of kda_prefill on the same inputs
 * (equal-length batches, per-channel gate).
 *
 *   q, k, v, alpha, beta, initial_state  as for kda_prefill (read)
 *   d_o            [B, T, H, d_v] qkv_dtype: gradient of o (read)
 *   d_final_state  [B, H, d_k, d_v] float32 or NULL (zero) (read)
 *   dq, dk, dalpha [B, T, H, d_k] float32 (written)
 *   dv             [B, T, H, d_v] float32 (written)
 *   dbeta          [B, T, H] float32 (written; 4-byte aligned suffices)
 *   d_initial_state[B, H, d_k, d_v] float32 or NULL (not written)
 *   workspace      device scratch of kda_prefill_backward_workspace_bytes(...)
 *                  bytes, 16-byte aligned, owned by the caller: for every
 *                  64-token chunk of every sequence and head, the state before
 *                  it, the state gradient after it (4 d_k d_v bytes each), its
 *                  chunk tables (about 129 KB for d_k = 128) and four 64 x d_v
 *                  fp32 work tiles (1 KB per value column). Calls sharing
 *                  a workspace must not overlap.
 *
 * Every gradient is float32 whatever qkv_dtype is. With float32 inputs the
 * arithmetic has fp32 accuracy (CUDA cores, and tensor-core products with
 * every operand split into two tf32 parts); with bfloat16 inputs the
 * tensor-core products are single tf32 products (about 1e-3 relative, well
 * inside the bf16 tolerance). Each gradient element is written once by one
 * thread, so two calls on the same inputs give the same bits. Errors as for
 * kda_prefill; a missing or short workspace returns KDA_ERR_WORKSPACE before
 * anything runs.
 */
kda_status_t kda_prefill_backward(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                  const float *alpha, const float *beta, const float *initial_state,
                                  const void *d_o, const float *d_final_state, float *dq, float *dk, float *dv,
                                  float *dalpha, float *dbeta, float *d_initial_state, int B, int T, int H,
                                  int d_k, int d_v, void *workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_prefill_backward_gate - kda_prefill_backward with a gate kind (see
 * kda_gate_t): alpha and dalpha are [B, T, H, d_k] (CHANNEL), [B, T, H]
 * (SCALAR: the gradient of the one gate a token-head has, i.e. the sum over
 * the channels of the per-channel gradient) or unused and NULL-able (NONE).
 * Everything else as kda_prefill_backward (same workspace).
 */
kda_status_t kda_prefill_backward_gate(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                       const float *alpha, kda_gate_t gate, const float *beta,
                                       const float *initial_state, const void *d_o, const float *d_final_state,
                                       float *dq, float *dk, float *dv, float *dalpha, float *dbeta,
                                       float *d_initial_state, int B, int T, int H, int d_k, int d_v,
                                       void *workspace, size_t workspace_bytes, kda_stream_t stream);

/* Workspace bytes kda_prefill_backward needs (0 for invalid arguments). */
size_t kda_prefill_backward_workspace_bytes(int B, int T, int H, int d_k, int d_v);

/*
 * kda_varlen_prefill_backward - the gradients of kda_varlen_prefill (N
 * sequences packed along the token axis by cu_seqlens, each with its own
 * initial state and chunk grid), with a gate kind as in
 * kda_prefill_backward_gate. Layouts as kda_varlen_prefill; the gradients
 * have the layouts of their inputs ([T_total, H, ...]; d_initial_state
 * [N, H, d_k, d_v]). Every sequence's gradients are those of
 * kda_prefill_backward_gate on that sequence alone, bit for bit.
 * cu_seqlens (DEVICE) is checked on the device: on a bad one device_status
 * (DEVICE int32, nullable) receives KDA_DEV_BAD_CU_SEQLENS and nothing is
 * written; otherwise KDA_DEV_OK. workspace: kda_varlen_prefill_backward_
 * workspace_bytes(N, T_total, H, d_k, d_v) bytes, 16-byte aligned.
 */
kda_status_t kda_varlen_prefill_backward(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                         const float *alpha, kda_gate_t gate, const float *beta,
                                         const float *initial_state, const void *d_o, const float *d_final_state,
                                         float *dq, float *dk, float *dv, float *dalpha, float *dbeta,
                                         float *d_initial_state, const int32_t *cu_seqlens, int N, int T_total,
                                         int H, int d_k, int d_v, void *workspace, size_t workspace_bytes,
                                         int32_t *device_status, kda_stream_t stream);

/* Workspace bytes kda_varlen_prefill_backward needs (0 for invalid arguments). */
size_t kda_varlen_prefill_backward_workspace_bytes(int N, int T_total, int H, int d_k, int d_v);

/*
 * kda_selftest_bounded_wait - diagnostic with no counterpart in the method:
 * runs the tensor-core prefill on one bf16 sequence of one head (B = H = 1,
 * d_k = d_v = 128, T tokens, zero initial state; tensors as for kda_prefill)
 * with its state chain made to wait, at chunk `stall_chunk`, on a barrier
 * that nothing ever completes. Every wait of the kernel is bounded: this one
 * gives up after about a second, the kernel's other groups give up on the
 * waits that depended on it, the kernel records a nonzero device error word
 * (see kda_device_errors) and returns. Its o and final_state are then
 * invalid. It exists so that a test can show that a stuck wait ends in an
 * error status, with the GPU context still usable, instead of a hang.
 * stall_chunk must lie in [0, ceil(T / 64)); KDA_ERR_INVALID_ARG otherwise.
 */
kda_status_t kda_selftest_bounded_wait(const void *q, const void *k, const void *v, const float *alpha,
                                       const float *beta, void *o, float *final_state, int T, int stall_chunk,
                                       kda_stream_t stream);

/* Message of the last failing call on this thread ("" if none). */
const char *kda_last_error(void);

/* ABI version of this header (incremented on incompatible changes). */
int kda_abi_version(void);

#define KDA_ABI_VERSION 1

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
