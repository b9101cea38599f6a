/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunked prefill for Kimi Delta
 * Attention (KDA).
 *
 * The operation. KDA keeps one fixed-size recurrent state per (sequence,
 * head) in place of a growing key-value cache, and every token updates it
 * ("Kimi K3 開源基礎設施", section "FlashKDA"; "Kimi K3 的三個系統設計",
 * section "第一個設計"). The update is the gated delta rule with a decay per
 * key channel:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * with S a K x V fp32 matrix (row = key channel). Prefill computes it in
 * 16-token chunks with two kernels of different parallelism, a
 * token-parallel intra-chunk kernel and a recurrent inter-chunk kernel
 * ("Kimi K3 的三個系統設計", section "為什麼 FlashKDA 選擇 16-token chunks"),
 * over fixed-length or packed variable-length batches with K = V = 128
 * ("MoonEP / FlashKDA / AgentENV" release note, section "MoE通信とアテンション").
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must be CUDA device memory (or
 *     managed memory) on the CURRENT device; the caller owns them. The
 *     library never frees them and holds none of them after the stream work
 *     the call enqueued has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is enqueued on it; no entry point but
 *     kda_last_device_error() blocks the host.
 *   - Errors found from the arguments alone are returned before anything
 *     is enqueued and leave every output untouched.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL_ARG = -1,          /* a required pointer is NULL */
    KDA_ERR_BAD_SHAPE = -2,         /* B, T, H, N inconsistent or out of range */
    KDA_ERR_UNSUPPORTED_DIM = -3,   /* K or V is not 128 */
    KDA_ERR_MISALIGNED = -4,        /* a pointer breaks the alignment rule below */
    KDA_ERR_BAD_CU_SEQLENS = -5,    /* (device) cu_seqlens not 0..T nondecreasing */
    KDA_ERR_CUDA = -6,              /* a CUDA runtime call failed */
    KDA_ERR_DEVICE_TIMEOUT = -7,    /* (device) a bounded wait inside a kernel ran out */
    KDA_ERR_NO_DEVICE_SUPPORT = -8, /* current device is not sm_103 */
    KDA_ERR_ALIAS = -9,             /* out or final_state overlaps an input */
    KDA_ERR_GATE_RANGE = -10,       /* (device) log decay rose by more than 80 inside a chunk */
    KDA_ERR_CAPTURE = -11,          /* workspace must grow while the stream is capturing */
    KDA_ERR_WRONG_DEVICE = -12,     /* a buffer or the stream belongs to another device */
    KDA_ERR_NOT_DEVICE_MEMORY = -13, /* a pointer is not CUDA device (or managed) memory */
    KDA_ERR_SCRATCH_LIMIT = -14,    /* kda_chunk_prefill_noalloc: the call needs more scratch
                                       than its fixed 64 MiB array holds */
    KDA_ERR_BAD_FLAGS = -15         /* a preprocessing flag bit this library does not know */
} kda_status;

/*
 * Input preprocessing done inside the kernels (the `flags` argument of
 * kda_chunk_prefill_ex and kda_decode_step). The pages leave the production
 * of q, k and g to the model; these let a caller hand over raw projections and
 * skip a separate pass over them.
 *   KDA_PRE_NORM_QK      q and k are raw: the kernels use x / sqrt(sum x^2 + 1e-6)
 *                        over the 128 channels of each (token, head)
 *   KDA_PRE_GATE_LOGITS  g holds gate logits x: the per-token log decay is
 *                        logsigmoid(x) = -log(1 + exp(-x))
 */
enum { KDA_PRE_NORM_QK = 1, KDA_PRE_GATE_LOGITS = 2 };

/*
 * kda_chunk_prefill -- chunked KDA prefill over a batch of sequences.
 *
 * Layout (all row-major, tokens of all sequences packed back to back):
 *   q, k      device, bf16  [B*T, H, K]   (the method expects L2-normalised rows)
 *   v         device, bf16  [B*T, H, V]
 *   g         device, fp32  [B*T, H, K]   per-token log decay (<= 0), NOT cumulated
 *   beta      device, fp32  [B*T, H]      in (0, 1)
 *   initial_state device, fp32 [N, H, K, V] or NULL (= zero state);
 *             element [n,h,i,j] is S[key i][value j]
 *   cu_seqlens device, int32 [N+1] or NULL. NULL: N = B sequences of T tokens
 *             each. Non-NULL: B must be 1, sequence n holds tokens
 *             [cu[n], cu[n+1]); cu[0] = 0, cu[N] = T, nondecreasing (empty
 *             sequences allowed). Checked on the device: a violation makes
 *             the kernels skip all work and kda_last_device_error() report
 *             KDA_ERR_BAD_CU_SEQLENS.
 *   B, T, H, K, V, N  sizes; K = V = 128 only; H >= 1; T >= 0; N >= 1;
 *             B*T*H*128 < 2^40.
 *   scale     multiplies o (1/sqrt(K) is the usual choice).
 *   out       device, bf16 [B*T, H, V], written for every token.
 *             With zero tokens (B*T == 0) q, k, v, g, beta and out may be NULL.
 *   final_state device, fp32 [N, H, K, V] or NULL (= not written); may equal
 *             initial_state (updated in place).
 *   stream    cudaStream_t as void*.
 *
 * Alignment: q, k, v, g, out, initial_state, final_state 16-byte aligned;
 * beta and cu_seqlens 4-byte aligned.
 *
 * Gate range: g may be any finite log decay <= 0. Chunks whose per-channel
 * cumulative log decay stays in [-80, 80] use factored exponentials
 * exp(G_r) exp(-G_i); the others take an exact per-pair form (slower, same
 * results to rounding). Positive g is allowed as long as the cumulative log
 * decay does not rise by more than 80 between two points of a 16-token chunk
 * (counting the chunk start as 0); beyond that exp() leaves fp32's range and
 * the device flags KDA_ERR_GATE_RANGE (results then unspecified).
 *
 * Workspace: the library keeps one scratch buffer per (device, stream),
 * grown stream-ordered (cudaMallocAsync / cudaFreeAsync) when a call needs
 * more (17,412 B per chunk-head: its record and one list entry). A
 * fixed-length call on the 16-token path whose sequences have at least 64
 * chunks and with 4*N*H <= (SM count - 4) runs a segment-parallel scan with
 * P = 3*(SM count - 4) / (2*N*H) segments (at most 16, at least 16 chunks per
 * segment; or the P set by kda_set_scan_segments): every sequence is cut
 * into P segments whose affine state maps are built in parallel, a short
 * serial combine gives each segment's entry state, and all segments are
 * replayed side by side (same results to rounding; not with an in-place
 * state). It reserves (3P - 5) * N*H*64 KiB more. Concurrent calls on
 * different streams never share scratch. Growing is refused with KDA_ERR_CAPTURE
 * while the stream is being captured into a graph: make one call of the
 * largest size before capturing. kda_workspace_release() frees them.
 *
 * Returns KDA_OK once the work is enqueued, or a synchronous error. Errors
 * found on the device are reported by kda_last_device_error().
 */
KDA_API kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *initial_state,
                             const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
                             int64_t K, int64_t V, int64_t N, float scale, void *out,
                             float *final_state, void *stream);

/*
 * kda_chunk_prefill_ex -- kda_chunk_prefill with input preprocessing:
 * `flags` is a bitwise OR of KDA_PRE_* (0 = kda_chunk_prefill exactly). An
 * unknown bit returns KDA_ERR_BAD_FLAGS. Everything else, including the
 * gate range of the resulting log decays, is as for kda_chunk_prefill.
 */
KDA_API kda_status kda_chunk_prefill_ex(const void *q, const void *k, const void *v,
                                        const float *g, const float *beta,
                                        const float *initial_state, const int32_t *cu_seqlens,
                                        int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                                        int64_t N, float scale, int flags, void *out,
                                        float *final_state, void *stream);

/*
 * kda_chunk_prefill_noalloc -- the same computation, arguments and results
 * as kda_chunk_prefill, for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for users of
 * the library whose code may not call cudaMalloc/cudaMallocAsync (directly or
 * through this library): a host framework that owns all device allocations,
 * a serving loop that must not enter the driver's allocator on its hot path,
 * or a sandboxed plug-in. It allocates nothing. Its scratch is one
 * fixed-size device array inside the library (64 MiB, held on every GPU that
 * loads the library until the process exits). The call holds at once a
 * 256-byte flag block, the chunk-offset table of a packed batch ((N+1)*4 B),
 * every chunk record (17,408 B per 16-token chunk per head) and a 4-byte
 * list entry per chunk-head, each part rounded up to 256 B; a call that needs
 * more than 64 MiB (about 3850 chunk-heads) returns KDA_ERR_SCRATCH_LIMIT
 * before enqueuing anything. All calls share that array: calls whose GPU
 * work overlaps (e.g. on two streams) race and give wrong results. The first
 * call on a device does a one-time set-up with that device current (no
 * allocation); make it before any stream capture (a first call on a
 * capturing stream returns KDA_ERR_CAPTURE). Uncaptured calls check their
 * pointers and stream like kda_chunk_prefill (KDA_ERR_NOT_DEVICE_MEMORY,
 * KDA_ERR_WRONG_DEVICE). Device errors of this entry point are reported by
 * kda_last_device_error() like those of the others.
 */
KDA_API kda_status kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v,
                                             const float *g, const float *beta,
                                             const float *initial_state,
                                             const int32_t *cu_seqlens, int64_t B, int64_t T,
                                             int64_t H, int64_t K, int64_t V, int64_t N,
                                             float scale, void *out, float *final_state,
                                             void *stream);

/*
 * kda_decode_step -- one new token for each of N sequences: the KDA state
 * update applied once per (sequence, head). The pages describe the state as
 * fixed-size and updated for every new token ("Kimi K3 的三個系統設計",
 * section 第一個設計); this is that step, batched:
 *
 *   S <- (I - beta k k^T) Diag(exp(g)) S + beta k v^T,   o = scale * S^T q
 *
 * with the post-update S, exactly the prefill recurrence at T = 1.
 *
 *   q, k, v      bf16 [N, H, 128], device, 16-byte aligned
 *   g            fp32 [N, H, 128] per-token log decay (any value; the
 *                exponentials are exact per channel, no range limit)
 *   beta         fp32 [N, H]
 *   state_in     fp32 [N, H, 128 (K), 128 (V)] or NULL (zero state)
 *   state_out    fp32 [N, H, 128, 128], written; may be state_in itself
 *                (in place) but may not overlap it otherwise
 *   N, H         sequences and heads (N * H < 2^31); K = V = 128 only
 *   flags        KDA_PRE_* bits (0: q, k, g used as given), as for
 *                kda_chunk_prefill_ex
 *   out          bf16 [N, H, 128], written; may not overlap any input or state
 *   stream       cudaStream_t (NULL = legacy default stream)
 *
 * Allocates nothing and reads no workspace: each (sequence, head) is one CTA
 * that reads its state once and writes it once. Returns KDA_OK once the work
 * is enqueued, or a synchronous error (the outputs are then untouched). It
 * has no device-side error conditions.
 */
KDA_API kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *g,
                                   const float *beta, const float *state_in, float *state_out,
                                   int64_t N, int64_t H, int64_t K, int64_t V, float scale,
                                   int flags, void *out, void *stream);

/*
 * kda_chunk_prefill_backward -- gradients of kda_chunk_prefill (training).
 * The pages say that K3 trains with KDA ("Kimi K3 開源基礎設施"); this is the
 * reverse mode of the same map, for a loss L with dL/do = d_out and
 * dL/d(final_state) = d_final_state:
 *
 *   dq, dk, dg  fp32 [B*T, H, 128]  dL/dq, dL/dk, dL/dg (g = the log decay)
 *   dv          fp32 [B*T, H, 128]  dL/dv
 *   dbeta       fp32 [B*T, H]       dL/dbeta
 *   d_initial_state  fp32 [N, H, 128, 128] or NULL (not written):
 *               dL/d(initial_state) (the gradient of a zero state when
 *               initial_state is NULL)
 *
 * Inputs exactly as for kda_chunk_prefill (q, k, v bf16; g, beta fp32;
 * initial_state, cu_seqlens, B, T, H, K, V, N, scale), plus
 *   d_out          bf16 [B*T, H, 128], device
 *   d_final_state  fp32 [N, H, 128, 128] or NULL (= 0)
 * Outputs are device memory the caller owns, every element written; none may
 * overlap an input or another output. Alignment: 16 bytes for every array
 * but beta, dbeta and cu_seqlens (4 bytes). No input preprocessing: q, k
 * and g are used as given. Any finite g.
 *
 * Method: one CTA per (sequence, head) walks the sequence backwards token
 * by token, the state recomputed from checkpoints taken every 16 tokens.
 * Workspace (the call's stream's, as for the prefill): 64 KiB per 16-token
 * chunk per head plus 1 MiB per CTA of the persistent kernel, min(N * H,
 * 1024) of them. Errors as for the prefill
 * (bad cu_seqlens contents are flagged on the device, see
 * kda_last_device_error).
 */
KDA_API kda_status kda_chunk_prefill_backward(const void *q, const void *k, const void *v,
                                              const float *g, const float *beta,
                                              const float *initial_state,
                                              const int32_t *cu_seqlens, int64_t B, int64_t T,
                                              int64_t H, int64_t K, int64_t V, int64_t N,
                                              float scale, const void *d_out,
                                              const float *d_final_state, float *dq, float *dk,
                                              float *dv, float *dg, float *dbeta,
                                              float *d_initial_state, void *stream);

/* Static text for a status code (never NULL). */
KDA_API const char *kda_status_string(kda_status status);

/*
 * Synchronises `stream`, then returns and clears the first error a kernel
 * of this library recorded on the current device since the last call
 * (KDA_OK if none). Device errors are sticky per device, not per stream;
 * this reads both the library's error word and that of the fixed array of
 * kda_chunk_prefill_noalloc (if that entry point has run on the device).
 */
KDA_API kda_status kda_last_device_error(void *stream);

/*
 * Frees every cached workspace buffer of the current device after
 * synchronising the device. Safe to call at any time no call of this
 * library is in flight on the device.
 */
KDA_API kda_status kda_workspace_release(void);

/* Workspace bytes a call with these sizes needs (0 on bad sizes). Host only. */
KDA_API int64_t kda_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t N, int has_cu_seqlens);

/* The same for kda_chunk_prefill_backward with the gradient form set by
 * kda_set_backward_impl: chunked (default): 256 B of flags, the packed chunk
 * offsets, then per 16-token chunk per head 17,408 B of record, 4 B of list
 * entry (rounded up to 256 B in all), 1,280 B of (I + A)^-1 and 64 KiB of
 * bf16 states;
 * token-serial: 256 B of flags, the packed chunk offsets, 64 KiB per
 * 16-token chunk per head and 1 MiB for each of min(N * H, 1024) state
 * rings. Both entry points share the stream's buffer, grown to the larger. */
KDA_API int64_t kda_backward_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t N,
                                             int has_cu_seqlens);

/*
 * Measurement hook (per host thread). kda_stage_timing_begin(max_calls)
 * creates 3*max_calls timing events on the current device; each of the next
 * max_calls kda_chunk_prefill() calls of this thread records one before the
 * intra-chunk kernel, one between it and the recurrent kernel, and one after
 * the recurrent kernel, on the call's stream. kda_stage_timing_end()
 * waits for those events, writes the mean milliseconds per call of the
 * intra-chunk stage (prologue excluded; the intra-chunk kernel and the exact
 * form of the chunks outside the factored range) and of the recurrent stage, and the
 * number of calls timed, then frees the events. Host pointers; NULL outputs
 * are skipped. Errors: KDA_ERR_BAD_SHAPE for max_calls < 1, KDA_ERR_CUDA.
 */
KDA_API kda_status kda_stage_timing_begin(int max_calls);
KDA_API kda_status kda_stage_timing_end(double *intra_ms, double *recurrent_ms, int *calls);

/*
 * Selects the gradient form for later kda_chunk_prefill_backward calls
 * (process-wide, host only): 0 (default) = chunked: the forward's
 * intra-chunk kernels build the chunk records and each chunk's (I + A)^-1
 * (fp32), the forward chain runs again
 * keeping every chunk's entry state (bf16), a reverse chain over the chunks
 * keeps every chunk's dL/d(exit state) (bf16) and writes dL/d(initial
 * state), and a chunk-parallel kernel computes dq, dk, dv, dg and dbeta
 * (workspace: per chunk-head 17,408 B of record, 4 B of list entry, 1,280 B
 * of (I + A)^-1 and 64 KiB of states); 1 = the token-serial first form. Both compute the same
 * gradients to rounding. Other values: KDA_ERR_BAD_SHAPE.
 */
KDA_API kda_status kda_set_backward_impl(int impl);

/*
 * Test hook for the device-timeout report (process-wide, host only; not for
 * production use). For later calls on the 16-token path, the record producer
 * of every recurrent CTA issues no copy for chunk `chunk` of its sequence or
 * any later one, and both roles of that kernel give up a wait after `wait_ns`
 * nanoseconds (0: the default of 2 s). The consumers' wait for that chunk
 * then runs out: they record KDA_ERR_DEVICE_TIMEOUT in the device error word
 * and leave (outputs from that chunk on and the final state are then
 * unspecified). Every copy the producer did issue is waited for, so none is
 * in flight when a CTA exits. chunk = -1 turns the hook off (the default).
 * chunk < -1 or wait_ns < 0: KDA_ERR_BAD_SHAPE.
 */
KDA_API kda_status kda_test_stall_recurrent(int chunk, int64_t wait_ns);

/*
 * Segments of the segment-parallel scan for later fixed-length calls on the
 * 16-token path (process-wide, host only): 0 (default) = chosen from the SM
 * count as described for kda_chunk_prefill, 1 = off (one chain per
 * sequence), P >= 2 = P segments (fewer when the sequence has fewer chunks
 * than P, or when that leaves a segment empty). Values outside [0, 4096]:
 * KDA_ERR_BAD_SHAPE. Takes effect for later calls (the workspace grows if
 * needed).
 */
KDA_API kda_status kda_set_scan_segments(int segments);

/*
 * Selects the chunk size and kernels for later calls (process-wide, host
 * only): 1 (default) = 16-token chunks, the intra-chunk kernel and then the
 * warp-level MMA recurrent kernel (state in registers, one CTA per
 * (sequence, head, 64 value channels)); 3 = 64-token chunks on the
 * 5th-generation tensor core, an intra-chunk kernel (tcgen05 Gram, W and U
 * products) and then a recurrent kernel (state in tensor memory, one CTA per
 * (sequence, head)); 4 = the 64-token kernels in one cooperative launch,
 * records passed through an L2-resident ring (3 when the heads leave fewer
 * than 16 SMs to the record builders). All compute the same result to
 * rounding. Other values: KDA_ERR_BAD_SHAPE.
 */
KDA_API kda_status kda_set_recurrent_impl(int impl);

/* Library build string: version and target architecture. Host only. */
KDA_API const char *kda_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
