/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library.
 *
 * The operator.  Per head, KDA keeps a state S in R^{d_k x d_v} and, for every
 * token t, applies
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = S_t^T q_t,
 *
 * with alpha_t in (0,1)^{d_k} a forget gate per key channel and beta_t a
 * scalar write strength ("Kimi K3" blog, section "Kimi Delta Attention"; the
 * same update in words on the "LLM architecture at trillion scale" page,
 * section "The KDA update, in plain words").  The gate is passed as
 * log_alpha = ln(alpha_t), expected in [-5, 0): the log-decay bound stated on
 * that page.  Values outside it are computed but not guaranteed to meet the
 * accuracy target.  The tightest case of the bf16 tensor-core path is the
 * no-decay end of the range (log_alpha = -1e-4 on every channel, the gate's
 * upper clamp), where the state carries each chunk's operand rounding through
 * the whole sequence: over 8192 tokens and 32 heads the output error is about
 * 4.8e-3 with beta = 1 on every token and 5.0e-3 with beta drawn by sigmoid,
 * relative to max|o|, against the 5e-3 bf16 target (in that range the chunk
 * prep feeds its Gram operands to the tensor cores as f16).  The fp32
 * CUDA-core path stays well inside it (about 3e-3).
 *
 * Two entry points compute it:
 *   kda_prefill -- many tokens at once in the chunked form ("Kimi K3: the
 *                  manos, the mythos, the legendos", section "FlashKDA
 *                  Algorithm"), returning every o_t and the final state;
 *   kda_decode  -- one token per sequence, updating an fp32 state in place
 *                  (the per-token form of the same section).
 *
 * Conventions for every call
 *   - All tensor arguments are caller-owned, contiguous, row-major DEVICE
 *     pointers (cu_seqlens_host is the one host pointer).  The library never
 *     allocates device memory and never synchronises the stream, except in
 *     kda_get_last_device_status and once per device in the first long
 *     tensor-core prefill (below).
 *   - Work is enqueued on `stream` (0 = the legacy default stream).  A call
 *     returns once the work is enqueued.  A long tensor-core prefill (the
 *     longest sequence at least 1024 chunks, its state pass on at most half
 *     of the SMs) forks part of its work onto an internal high-priority
 *     stream of the library (created once per device, kept until exit) and
 *     joins it back into `stream` with events before returning, so ordering
 *     on `stream` holds.  The first such call on a device, unless `stream`
 *     is being captured into a graph, also runs a ~10 us kernel that finds
 *     which SM ids the device has (32 bytes of the workspace) and waits for
 *     it on `stream`; later calls reuse the result.
 *   - Arguments are checked before anything is launched; a failed check
 *     returns an error and launches nothing.  A launch failure returns
 *     KDA_ERR_CUDA.  Faults detected inside a kernel (a wait that ran out of
 *     time) are recorded in a device status word read by
 *     kda_get_last_device_status.
 *   - Supported shapes: d_k, d_v in {32, 64, 128}; chunk in {16, 32, 64}.
 *     KDA_BF16 with d_k = d_v = 128 and chunk = 64 runs on the tcgen05
 *     tensor-core path; every other combination runs on the fp32 CUDA-core
 *     chunked path.  Both are GPU kernels; there is no CPU path.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad cu_seqlens, ... */
    KDA_ERR_UNSUPPORTED = 2,  /* shape / dtype / chunk combination not built     */
    KDA_ERR_WORKSPACE = 3,    /* workspace missing, too small or misaligned      */
    KDA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed             */
    KDA_ERR_TIMEOUT = 5,      /* a kernel gave up waiting (device status only)    */
    KDA_ERR_PRECONDITION = 6, /* debug library: an input outside its stated range
                                 (device status only)                             */
    KDA_ERR_DEVICE_CHECK = 7  /* debug library: a kernel found an index outside its
                                 buffer and skipped the access (device status)    */
} kda_status;

typedef enum kda_dtype {
    KDA_FP32 = 0,             /* q, k, v and O are float                          */
    KDA_BF16 = 1              /* q, k, v and O are bfloat16 (raw 16-bit storage)  */
} kda_dtype;

/*
 * Bytes of device workspace kda_prefill needs for this problem.  0 means none
 * (the CUDA-core path).  The figure depends only on the arguments, and it
 * assumes the worst case of one partial chunk per sequence, so it is valid for
 * any cu_seqlens with these n_seq and T_total.
 */
KDA_API size_t kda_prefill_workspace_size(int n_seq, int T_total, int H, int dk, int dv,
                                  int chunk, kda_dtype dtype);

/*
 * Chunked prefill over a packed batch of variable-length sequences.
 *
 * Computes, for each sequence n and head h independently, the recurrence above
 * over the sequence's tokens, starting from S0[n,h], and returns o_t for every
 * token and the final state.  The chunked matrix form it evaluates is the one
 * of "Kimi K3: the manos, the mythos, the legendos", section "FlashKDA
 * Algorithm" (cumulative decay, Q_decay / K_decay / K_restore, the UT
 * transform U = (I + L)^{-1} Diag(beta)(V - K_decay S_in),
 * O = Q_decay S_in + M_qk U, S_out = Diag(a_last) S_in + K_restore^T U).
 *
 * q, k       [T_total, H, dk]  dtype
 * v          [T_total, H, dv]  dtype
 * log_alpha  [T_total, H, dk]  float, natural log of the gate
 * beta       [T_total, H]      float
 * S0         [n_seq, H, dk, dv] float, or NULL for zero initial states
 * cu_seqlens [n_seq + 1] int32 device array of token offsets (0 = cu[0] <=
 *            cu[1] <= ... <= cu[n_seq] = T_total), or NULL for n_seq
 *            sequences of equal length T_total / n_seq (which must divide).
 * cu_seqlens_host  optional host copy of cu_seqlens (same values).  When
 *            given it is validated and used to size the launch exactly; when
 *            NULL a device cu_seqlens is trusted (lengths are clamped on the
 *            device so that no access leaves the arrays).
 * O          [T_total, H, dv]  dtype, written for every token; must not alias
 *            an input.
 * S_final    [n_seq, H, dk, dv] float, or NULL.  May alias S0 exactly.
 * workspace  device memory of at least kda_prefill_workspace_size(...) bytes,
 *            256-byte aligned (may be NULL when that size is 0).  Its contents
 *            on entry do not matter; the call owns it until the work completes.
 * Sequences of length 0 are allowed (their S_final is S0).
 * On the tensor-core path (bf16, dk = dv = 128, chunk 64) q, k, v, log_alpha
 * and O must be 16-byte aligned; otherwise KDA_ERR_INVALID_ARG.
 */
KDA_API kda_status kda_prefill(const void* q, const void* k, const void* v,
                       const float* log_alpha, const float* beta, const float* S0,
                       const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                       int n_seq, int T_total, int H, int dk, int dv, int chunk,
                       kda_dtype dtype, void* O, float* S_final,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_prefill that also saves the recurrent state at coarse positions, for
 * prefix caching: a linear-attention layer can only resume a cached prefix
 * from a stored state, so serving stacks keep the state every so many tokens
 * ("Kimi K3: the manos, the mythos, the legendos", section "KDA Prefix Cache
 * Management"; the "LLM architecture at trillion scale" page, section "6. Deep
 * dive: what this means for serving").
 *
 * Arguments as kda_prefill, plus:
 * ckpt_every     positive multiple of chunk: a checkpoint is the state after
 *                the first m * ckpt_every tokens of a sequence (m = 1, 2, ...,
 *                as long as m * ckpt_every <= its length)
 * ckpt           [ckpt_capacity, H, dk, dv] float device array, 16-byte
 *                aligned (else KDA_ERR_INVALID_ARG); checkpoint m of
 *                sequence n goes to index sum_{n' < n} floor(len_n' /
 *                ckpt_every) + m - 1
 * ckpt_capacity  number of checkpoints ckpt holds; when the lengths are known
 *                on the host (cu_seqlens_host, or equal lengths) a smaller
 *                capacity than needed is KDA_ERR_INVALID_ARG, otherwise
 *                checkpoints past the capacity are not written.
 */
KDA_API kda_status kda_prefill_ckpt(const void* q, const void* k, const void* v,
                            const float* log_alpha, const float* beta, const float* S0,
                            const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                            int n_seq, int T_total, int H, int dk, int dv, int chunk,
                            kda_dtype dtype, void* O, float* S_final, int ckpt_every,
                            float* ckpt, int ckpt_capacity, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/*
 * Size of the fixed device array that kda_prefill_noalloc uses as its
 * workspace (bytes).  Under CUDA's lazy module loading (the default) a device
 * reserves it when the first kda_prefill_noalloc call on that device loads
 * the code that holds it, and keeps it until the process exits.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * kda_prefill without a caller-provided workspace.  The paper has no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory -- runtimes that own all device memory through their own fixed pool
 * and do not let libraries call cudaMalloc, plugin interfaces that give a
 * library only its inputs and outputs, and deployments whose memory footprint
 * is fixed at start-up.
 *
 * Same arguments and results as kda_prefill, minus (workspace,
 * workspace_bytes).  The workspace is a file-scope device array of
 * KDA_NOALLOC_SCRATCH_BYTES; the call allocates nothing.
 *   - Returns KDA_ERR_WORKSPACE, before launching anything, when
 *     kda_prefill_workspace_size(...) for the problem exceeds
 *     KDA_NOALLOC_SCRATCH_BYTES (e.g. more than about 500 chunk-head slots
 *     on the tensor-core path: H = 32 heads of ~900 tokens).
 *   - Every call looks up the array's device address on the current device
 *     (the device of the tensors must be current).  The first call on a
 *     device also loads the code that holds the array, which reserves its
 *     64 MiB there (KDA_ERR_CUDA if that fails): make that first call at
 *     start-up, before a fixed-pool runtime takes its pool and before any
 *     stream capture.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls that overlap
 *     on the GPU race on it: order them on one stream.
 */
KDA_API kda_status kda_prefill_noalloc(const void* q, const void* k, const void* v,
                               const float* log_alpha, const float* beta, const float* S0,
                               const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                               int n_seq, int T_total, int H, int dk, int dv, int chunk,
                               kda_dtype dtype, void* O, float* S_final, cudaStream_t stream);

/*
 * Fused parameter-free prologue.  The Kimi Linear layer L2-normalises q and k
 * before the operator ("Kimi K3: the manos, the mythos, the legendos",
 * section "Kimi Linear") and keeps the log-decay inside (-5, 0) ("LLM
 * architecture at trillion scale", section "The KDA update, in plain words").
 * The *_fused entries take those inputs before the activations and apply, in
 * fp32 inside the kernels, per (token, head):
 *   q <- q / sqrt(sum_i q_i^2 + 1e-6),  k <- k / sqrt(sum_i k_i^2 + 1e-6)
 *   log_alpha = clamp(-softplus(gate), -5, -1e-4)      (per key channel)
 *   beta = sigmoid(beta_logit)
 * and then compute exactly what kda_prefill / kda_decode compute.
 *
 * kda_prefill_fused: arguments as kda_prefill, with
 *   q, k        [T_total, H, dk] dtype, not normalised
 *   gate        [T_total, H, dk] float, pre-activation of the log-decay
 *   beta_logit  [T_total, H] float, pre-activation of beta
 * (workspace from kda_prefill_workspace_size, as for kda_prefill).
 */
KDA_API kda_status kda_prefill_fused(const void* q, const void* k, const void* v,
                             const float* gate, const float* beta_logit, const float* S0,
                             const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                             int n_seq, int T_total, int H, int dk, int dv, int chunk,
                             kda_dtype dtype, void* O, float* S_final, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_decode_fused: one decode step as kda_decode, with q, k [N, H, dk] not
 * normalised, gate [N, H, dk] and beta_logit [N, H] pre-activations (see
 * kda_prefill_fused for the prologue).
 */
KDA_API kda_status kda_decode_fused(const void* q, const void* k, const void* v,
                            const float* gate, const float* beta_logit, float* S, int N, int H,
                            int dk, int dv, kda_dtype dtype, void* o, cudaStream_t stream);

/*
 * One decode step for N independent sequences (one token each), the per-token
 * form u = beta (v - (D S)^T k), S <- D S + k u^T, o = S^T q of "Kimi K3: the
 * manos, the mythos, the legendos", section "FlashKDA Algorithm".
 *
 * q, k       [N, H, dk] dtype;  v [N, H, dv] dtype
 * log_alpha  [N, H, dk] float;  beta [N, H] float
 * S          [N, H, dk, dv] float, read and overwritten in place; 16-byte
 *            aligned (it moves as float4 vectors), else KDA_ERR_INVALID_ARG
 * o          [N, H, dv] dtype, written; must not alias an input.
 * N = 0 returns KDA_OK and launches nothing.
 */
KDA_API kda_status kda_decode(const void* q, const void* k, const void* v,
                      const float* log_alpha, const float* beta, float* S,
                      int N, int H, int dk, int dv, kda_dtype dtype, void* o,
                      cudaStream_t stream);

/*
 * Multi-token verify step for speculative decoding: the "LLM architecture at
 * trillion scale" page (section "6. Deep dive: what this means for serving")
 * has a draft model propose up to 7 tokens that the big model then checks.
 * For each of N sequences, K proposed tokens (K <= 16) are run through the
 * recurrence from the state S, every o_t is returned, and S is overwritten
 * with the state after the first commit_len[n] tokens only (0 leaves S as
 * it was; the rest of the proposal is not committed).
 *
 * q, k       [N, K, H, dk] dtype;  v [N, K, H, dv] dtype
 * log_alpha  [N, K, H, dk] float;  beta [N, K, H] float
 * S          [N, H, dk, dv] float, read, and written after commit_len tokens;
 *            16-byte aligned, else KDA_ERR_INVALID_ARG
 * commit_len [N] int32 device array, values clamped to [0, K]; NULL = K
 * K > 16 is KDA_ERR_UNSUPPORTED; N = 0 or K = 0 returns KDA_OK.
 * o          [N, K, H, dv] dtype, or NULL to skip the outputs
 * A typical use calls it twice: once with commit_len all 0 to get the
 * outputs, then, once the accepted lengths are known, with o = NULL and
 * commit_len = the accepted lengths.
 */
KDA_API kda_status kda_decode_multi(const void* q, const void* k, const void* v,
                            const float* log_alpha, const float* beta, float* S,
                            const int32_t* commit_len, int N, int K, int H, int dk, int dv,
                            kda_dtype dtype, void* o, cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the device status word:
 * KDA_OK, or KDA_ERR_TIMEOUT if a kernel since the last call gave up waiting
 * (its outputs are then incomplete), or KDA_ERR_CUDA if the synchronisation
 * itself failed.  The word is per device and shared by all streams.
 */
KDA_API kda_status kda_get_last_device_status(cudaStream_t stream);

/*
 * Check of the failure detection above (the pages have no counterpart; it
 * computes nothing of KDA): one kernel waits on an mbarrier that nothing
 * completes, with the same bounded wait the kernels use, for at most
 * `limit_cycles` SM clock cycles (0 ... ~4e9, the kernels' own limit of about
 * two seconds).  Afterwards kda_get_last_device_status returns KDA_ERR_TIMEOUT
 * and the device stays usable.  KDA_ERR_INVALID_ARG for a limit outside that
 * range, before anything is launched.
 */
KDA_API kda_status kda_check_wait_timeout(long long limit_cycles, cudaStream_t stream);

/*
 * Tracing hook.  While set, every kda_prefill / kda_decode call made from the
 * calling host thread records the given CUDA events (cudaEvent_t handles,
 * created by the caller) on its stream at the boundaries between the kernels
 * it launches, all on the caller's stream: event 0 before the first kernel;
 * for the tensor-core prefill, event 1 once every chunk-prep kernel has run
 * and event 2 when the state pass (which may run partly on an internal
 * stream, overlapped with later chunk preps, or as a segment scan of three
 * kernels for few long sequences) has finished on the caller's stream; for the
 * CUDA-core prefill and the decode, event 1 after their one kernel.  Events beyond
 * n_events are skipped.  Pass (NULL, 0) to stop.  Returns KDA_ERR_INVALID_ARG
 * for n_events < 0 or a NULL array with n_events > 0.  The array must stay
 * valid while the hook is set.  This exists so that a benchmark can time each
 * kernel with CUDA events on the stream the kernel runs on.
 */
KDA_API kda_status kda_set_trace_events(void* const* events, int n_events);

/*
 * Debug variant.  The library is also built as libkda_debug.so, compiled with
 * KDA_DEBUG: the same entry points with the same results, plus checks that the
 * release library leaves out for speed.
 *   - Precondition: before each kda_prefill, kda_prefill_ckpt,
 *     kda_prefill_noalloc, kda_decode and kda_decode_multi call, one pass over
 *     log_alpha records KDA_ERR_PRECONDITION in the device status word when a
 *     value lies outside [-5, 0] or is not a number.  That is the log-decay
 *     bound of "LLM architecture at trillion scale", section "The KDA update,
 *     in plain words", inside which the chunked form's staged decay factors
 *     stay finite and the accuracy target is stated; the call still computes.
 *     (The *_fused calls clamp the log-decay themselves and are not checked.)
 *   - Device checks: the tensor-core kernels check the workspace slots and
 *     segment indices they derive from the call's lengths against the sizes
 *     they were given; an index outside records KDA_ERR_DEVICE_CHECK and the
 *     access is skipped.  Nothing traps.
 * kda_get_last_device_status of the same library reports either code.
 * Returns 1 in the debug library, 0 in the release library.
 */
KDA_API int kda_debug_build(void);

/* Static, NUL-terminated description of a status code (never NULL). */
KDA_API const char* kda_status_string(kda_status status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
