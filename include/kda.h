/*
 * kda.h - C ABI of the GB300 (sm_103a) chunked forward pass of Kimi Delta
 * Attention (KDA).
 *
 * The operation (Kimi Delta Attention, arXiv:2510.26692, the paper cited by
 * the cuLA overview page on discuss.pytorch.kr, section "cuLA 소개"), per
 * sequence s and head h, for tokens t in order:
 *
 *   log alpha_t[k] = lower_bound * sigmoid(exp(A_log[h]) * (g[t,h,k] + dt_bias[h,k]))
 *   q_hat = q / sqrt(|q|^2 + 1e-6),  k_hat = k / sqrt(|k|^2 + 1e-6)
 *   beta_t = sigmoid(beta_logit[t,h])
 *   S_t = (I - beta_t k_hat k_hat^T) Diag(alpha_t) S_{t-1} + beta_t k_hat v_t^T   (S is K x V)
 *   o_t = scale * S_t^T q_hat
 *
 * The argument list and layouts follow the flash_kda.fwd parameter table on
 * the FlashKDA page (discuss.pytorch.kr, section "FlashKDA의 KDA 연산 구조"):
 * q/k/g bf16 [B,T,H,K], v bf16 [B,T,H,V], beta bf16 [B,T,H] logits, A_log
 * fp32 [H], dt_bias fp32 [H,K], lower_bound in [-5, 0], optional fp32
 * initial/final state [B,H,V,K]; the gate activation, q/k L2 norm and beta
 * sigmoid run inside the kernels (same section). Packed variable-length
 * batches pass int32 cu_seqlens (cuLA README mirror on shadowgraph.io,
 * "Quick Start" notes); then B must be 1 and the state has one row per
 * sequence. The computation is chunked (64 tokens per chunk, as in the FLA
 * and cuLA kernels described in section "Flash Linear Attention과 비교") and
 * split into a token-parallel prep kernel and a head-parallel recurrence
 * kernel (FlashKDA page, section "커널 퓨전(Kernel Fusion) 전략의 분리").
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers to contiguous row-major data,
 *     except where stated. The caller owns every buffer; the library keeps no
 *     pointer after a call returns. Work is enqueued on `stream` and is
 *     asynchronous: results are ready when the stream is synchronised.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns a status and enqueues nothing.
 *   - Errors found on the device (a malformed cu_seqlens) are recorded in a
 *     per-device status word and the kernels of that call return early
 *     without writing o; kda_get_device_status() reads and clears the word.
 *   - Nothing throws or aborts across this boundary.
 */
#ifndef KDA_GB300_KDA_H_
#define KDA_GB300_KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (a cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad alignment, bad scalar */
  KDA_ERR_UNSUPPORTED = 2,   /* head dims other than K, V in {64, 128} */
  KDA_ERR_WORKSPACE = 3,     /* workspace too small, or allocating it failed */
  KDA_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  KDA_ERR_DEVICE_STATUS = 5  /* the device recorded a data error (see below) */
} kda_status_t;

/* Device-side error codes reported through kda_get_device_status(). */
#define KDA_DEVICE_OK 0
#define KDA_DEVICE_BAD_CU_SEQLENS 1   /* cu_seqlens[0] != 0, decreasing, or cu_seqlens[N] != T */
#define KDA_DEVICE_WAIT_TIMEOUT 2     /* a bounded pipeline wait in a kernel gave up */
/*
 * The recurrence ended with a non-finite state for some (sequence, head): an
 * input was not finite, or a value went past the fp16 range (|x| > 65504) of
 * the recurrence's tensor-core operands. Those operands are the state S, the
 * residuals U = v - prediction and v itself, rounded to fp16 once per chunk;
 * an overflow there turns into inf / NaN, which the fp32 state keeps, so a
 * check of every (sequence, head)'s last state catches it. The check runs
 * whether or not final_state is requested. o of that (sequence, head) is then
 * not valid.
 */
#define KDA_DEVICE_NONFINITE 3

/* Tokens per chunk of the chunked algorithm. */
#define KDA_CHUNK 64

/*
 * Bytes of scratch memory kda_fwd() needs for a problem of this size.
 * num_seqs is the number of sequences N: B without cu_seqlens, the length of
 * cu_seqlens minus one with it. Returns 0 when the sizes are invalid.
 * The scratch holds, per chunk and head, what the prep kernel hands to the
 * recurrence kernel: the 128 x 64 fp16 matrix
 * [-(I+A)^{-1} diag(beta); P (I+A)^{-1} diag(beta)], the decayed keys and
 * queries khat Gamma, khat Gamma_last / Gamma and qhat Gamma (fp16, 64 x K
 * each) and the chunk decay Gamma_last (fp32, K), plus the varlen schedule:
 * about 64.5 KiB per chunk of 64 tokens and head at K = 128.
 */
KDA_API size_t kda_fwd_workspace_size(int B, int T, int H, int K, int V, int num_seqs);

/*
 * kda_fwd_workspace_size() for a call of kda_fwd_ex() with these flags: the
 * context-parallel flags (KDA_CP_OFF, KDA_CP_SEGMENTS(n)) change the scratch
 * the call needs; the other flags do not. varlen is nonzero when the call will
 * pass cu_seqlens (context parallelism then never applies). Returns 0 when the
 * sizes or flags are invalid. kda_fwd_workspace_size(...) is
 * kda_fwd_workspace_size_ex(..., 0, 0): enough for kda_fwd() in either mode.
 */
KDA_API size_t kda_fwd_workspace_size_ex(int B, int T, int H, int K, int V, int num_seqs, int varlen,
                                         uint32_t flags);

/*
 * KDA chunked forward.
 *
 *   q, k, g      bf16 [B,T,H,K]; g is the pre-activation gate.
 *   v            bf16 [B,T,H,V].
 *   beta         bf16 [B,T,H] logits (sigmoid applied inside).
 *   A_log        fp32 [H].
 *   dt_bias      fp32 [H,K], or NULL for zeros.
 *   lower_bound  finite, in [-5, 0].
 *   scale        finite output scale (usually K^-0.5).
 *   initial_state fp32 [N,H,V,K] (state[s,h,v,k] = S[k,v]) or NULL for zeros.
 *   final_state  fp32 [N,H,V,K] to receive the last state, or NULL. It may be
 *                the same pointer as initial_state (in-place update); any
 *                other overlap is not allowed.
 *   cu_seqlens   int32 [N+1] prefix offsets of packed sequences, or NULL. When
 *                set, B must be 1, T is the packed length, and N = num_seqs.
 *                Zero-length sequences are allowed (their state is copied).
 *   B, T, H, K, V  sizes; K and V in {64, 128}; T may be 0.
 *   num_seqs     N: equal to B when cu_seqlens is NULL.
 *   o            bf16 [B,T,H,V] output.
 *   workspace    device scratch of at least kda_fwd_workspace_size() bytes,
 *                256-byte aligned, or NULL to let the call allocate and free
 *                it stream-ordered (cudaMallocAsync / cudaFreeAsync).
 *   stream       the CUDA stream to enqueue on.
 *
 * Alignment: q, k, v, g, o, initial_state and final_state must be 16-byte
 * aligned; dt_bias 16-byte; beta 2-byte; cu_seqlens, A_log 4-byte. When T == 0 the
 * token tensors (q, k, v, g, beta, o) hold nothing and may be NULL.
 * Returns KDA_OK when the work was enqueued. Concurrent calls on different
 * streams are safe when each has its own workspace and outputs.
 */
KDA_API kda_status_t kda_fwd(const void *q, const void *k, const void *v, const void *g,
                     const void *beta, const float *A_log, const float *dt_bias,
                     float lower_bound, float scale, const float *initial_state,
                     float *final_state, const int32_t *cu_seqlens, int B, int T,
                     int H, int K, int V, int num_seqs, void *o, void *workspace,
                     size_t workspace_bytes, kda_stream_t stream);

/*
 * Variant flags of kda_fwd_ex() (bitwise OR; 0 is kda_fwd()):
 *
 *   KDA_GATE_PER_HEAD  one decay per token and head instead of per channel (the
 *                      gated delta rule, GDN, of the cuLA overview and FlashQLA
 *                      pages): g is bf16 [B,T,H] and dt_bias fp32 [H] (or NULL),
 *                      and every channel k of head h takes
 *                      log alpha_t = lower_bound * sigmoid(exp(A_log[h]) * (g[t,h] + dt_bias[h])).
 *                      Alignment: g 2-byte, dt_bias 4-byte.
 *   KDA_BETA_F32       beta holds fp32 logits [B,T,H] (the cuLA Quick Start
 *                      notes: beta in float32 or bfloat16). Alignment 4-byte.
 *   KDA_STATE_BF16     initial_state and final_state are bf16 instead of fp32
 *                      (the FlashKDA parameter table: bf16/fp32 state). The
 *                      state is carried in fp32 inside; only its load and store
 *                      change, the store rounding to nearest-even.
 *   KDA_STATE_KV       initial_state and final_state are laid out [N,H,K,V]
 *                      (state[s,h,k,v] = S[k,v], the layout of the cuLA usage
 *                      example) instead of [N,H,V,K].
 *   KDA_EXP2_POLY      an implementation option, not a variant of the operation:
 *                      the per-token, per-channel decays alpha = 2^(log2 alpha)
 *                      are evaluated by a polynomial on the FMA pipe instead of
 *                      the SFU exponential (the polynomial exponential of the
 *                      cuLA launch blog, section "Status & Roadmap"). Results agree within
 *                      the same tolerances; it is off by default because the
 *                      prep kernel measured slower with it on GB300.
 */
#define KDA_GATE_PER_HEAD 0x1u
#define KDA_BETA_F32 0x2u
#define KDA_STATE_BF16 0x4u
#define KDA_STATE_KV 0x8u
#define KDA_EXP2_POLY 0x10u

/*
 * Intracard context parallelism (the FlashKDA intracard CP of the cuLA README
 * mirror, section "Benchmarks"; the gate-driven intracard context parallelism
 * of the FlashQLA page, section "핵심 기능"), an implementation option that does
 * not change the operation. Each sequence is cut into segments of whole
 * chunks that run in parallel: a first pass runs every segment from a zero
 * state and also forms its K x K state transition, a small combine pass chains
 * the segments' start states, and a second pass reruns every segment from its
 * true start state. It costs up to about three times the recurrence work and
 * pays only when the plain recurrence leaves most SMs idle (few long
 * sequences and heads). Fixed-length batches only: with cu_seqlens it is never
 * used.
 *
 *   (default)            chosen per call from the sizes and the SM count, where
 *                        the library's estimate shows a clear gain.
 *   KDA_CP_OFF           never.
 *   KDA_CP_SEGMENTS(n)   always, with n segments per sequence, n in [2, 64]
 *                        (segments past the end of a short sequence are empty).
 * The workspace must then be sized by kda_fwd_workspace_size_ex() with the
 * same flags: segment states need (2 V + K) K fp32 values per (sequence,
 * segment, head).
 */
#define KDA_CP_OFF 0x20u
#define KDA_CP_SEGMENTS(n) ((((uint32_t)(n)) & 0xFFu) << 8)

/*
 * Stage timing hooks for kda_fwd_with_events(): CUDA events (cudaEvent_t,
 * created by the caller) recorded on `stream` at the stage boundaries. Any
 * member may be NULL. prep_start precedes the varlen schedule (if any) and
 * the prep kernel; prep_done separates the prep kernel from the recurrence
 * kernel; recur_done follows the recurrence kernel.
 * Without prep_done the recurrence kernel is launched to overlap the end of
 * the prep kernel (programmatic dependent launch: its blocks may take the SMs
 * the prep kernel frees, and wait on the GPU for it to finish before they
 * read anything), as kda_fwd() does; with prep_done it starts after the prep
 * kernel has finished, so that the event splits the time between the two.
 */
typedef struct {
  void *prep_start;
  void *prep_done;
  void *recur_done;
} kda_stage_events_t;

/*
 * kda_fwd() with stage events recorded for profiling (same arguments, same
 * results; `events` may be NULL, which makes it identical to kda_fwd()).
 * Defined by the same operation as kda_fwd(); the events only timestamp the
 * two kernels the chunked forward is split into (FlashKDA page, section
 * "커널 퓨전(Kernel Fusion) 전략의 분리").
 */
KDA_API kda_status_t kda_fwd_with_events(const void *q, const void *k, const void *v, const void *g,
                                         const void *beta, const float *A_log, const float *dt_bias,
                                         float lower_bound, float scale, const float *initial_state,
                                         float *final_state, const int32_t *cu_seqlens, int B, int T,
                                         int H, int K, int V, int num_seqs, void *o, void *workspace,
                                         size_t workspace_bytes, kda_stream_t stream,
                                         const kda_stage_events_t *events);

/*
 * kda_fwd_with_events() with variant flags (KDA_GATE_PER_HEAD, KDA_BETA_F32,
 * KDA_STATE_BF16, KDA_STATE_KV, above). The state pointers are untyped: fp32
 * or bf16 by KDA_STATE_BF16, [N,H,V,K] or [N,H,K,V] by KDA_STATE_KV; every
 * other argument, layout, alignment rule and error is that of kda_fwd(), except
 * where a flag states otherwise. Unknown flag bits give KDA_ERR_INVALID_ARG.
 * kda_fwd(...) is kda_fwd_ex(..., 0, ...) with events NULL.
 */
KDA_API kda_status_t kda_fwd_ex(const void *q, const void *k, const void *v, const void *g,
                                const void *beta, const float *A_log, const float *dt_bias,
                                float lower_bound, float scale, const void *initial_state,
                                void *final_state, const int32_t *cu_seqlens, int B, int T, int H,
                                int K, int V, int num_seqs, uint32_t flags, void *o, void *workspace,
                                size_t workspace_bytes, kda_stream_t stream,
                                const kda_stage_events_t *events);

/*
 * Diagnostic entry point: runs only the varlen schedule and the token-parallel
 * prep kernel of kda_fwd() and copies, for every chunk c (in sequence order,
 * chunk c of sequence s at index chunk_offset[s] + c, where chunk_offset is the
 * exclusive prefix sum of ceil(len_s / 64)) and head h, the fp16 matrix
 *   M[c,h] = [ -Tb ; P Tb ]  (128 x 64),  Tb = (I + A)^{-1} diag(beta)
 * into `chunk_mats` (device, fp16 [max_chunks][H][128][64], max_chunks =
 * kda_max_chunks(B, T, num_seqs)). A, P are the decay-weighted strictly lower
 * key-key and lower query-key chunk matrices. Rows and columns past the end
 * of a partial chunk are zero (their beta is taken as 0). Each 128 x 64 block
 * is stored in the 128-byte-swizzled order the recurrence kernel loads it in:
 * the 16-byte chunk c (8 values, columns 8c..8c+7) of row r sits at position
 * r * 8 + (c XOR (r mod 8)) of the block. Same arguments and errors as
 * kda_fwd() otherwise.
 */
KDA_API kda_status_t kda_debug_chunk_matrices(const void *q, const void *k, const void *g,
                                      const void *beta, const float *A_log,
                                      const float *dt_bias, float lower_bound,
                                      const int32_t *cu_seqlens, int B, int T, int H,
                                      int K, int num_seqs, void *chunk_mats,
                                      void *workspace, size_t workspace_bytes,
                                      kda_stream_t stream);

/*
 * kda_fwd() for callers that cannot allocate device memory. (This entry point
 * has no counterpart on the pages; it is a deployment convenience.)
 *
 * Who needs it: hosts that own all device memory themselves, such as a
 * serving runtime that reserves the whole GPU pool at start-up and gives a
 * kernel plug-in only its inputs and outputs, or a latency-critical path that
 * must not call cudaMalloc / cudaMallocAsync (they can synchronise the device
 * or grow a memory pool). Here the scratch that kda_fwd() would take from the
 * caller lives in a fixed array inside the library image, so the call
 * allocates nothing: it calls no cudaMalloc, cudaFree or allocating routine.
 *
 * Arguments, layouts and results are those of kda_fwd() without the
 * workspace pair; the caller still passes every input and output buffer.
 *
 * Limit: the problem must fit in KDA_NOALLOC_MAX_SCRATCH bytes of scratch,
 * i.e. kda_fwd_workspace_size_ex(B, T, H, K, V, num_seqs, cu_seqlens != NULL,
 * KDA_CP_OFF) <= KDA_NOALLOC_MAX_SCRATCH: this entry point never uses context
 * parallelism, whose segment states would take scratch away from the problem
 * (about 8 MiB per head per 8192 tokens at K = V = 128: B=1, T=8192 fits H = 1,
 * B=1, T=2048 fits H <= 7).
 * Larger problems are rejected with KDA_ERR_WORKSPACE before anything runs.
 * Every GPU that loads the library holds this array until the process exits.
 *
 * Set-up: the first call on each device looks up the device address of the
 * array (cudaGetSymbolAddress with that device current). Make that first call
 * before any stream capture on the device.
 *
 * Sharing: all calls on a device share the one array, and it keeps the last
 * call's contents (no call depends on it starting at zero). Calls whose work
 * overlaps on the GPU (for example on two streams at once) race on the array
 * and give wrong results: order them on one stream or synchronise between
 * them.
 */
#define KDA_NOALLOC_MAX_SCRATCH (16u * 1024u * 1024u)
KDA_API kda_status_t kda_fwd_noalloc(const void *q, const void *k, const void *v, const void *g,
                                     const void *beta, const float *A_log, const float *dt_bias,
                                     float lower_bound, float scale, const float *initial_state,
                                     float *final_state, const int32_t *cu_seqlens, int B, int T,
                                     int H, int K, int V, int num_seqs, void *o, kda_stream_t stream);

/*
 * The launch plan kda_fwd_ex() would use on the current device for these sizes
 * and flags: *n_segments gets the number of context-parallel segments per
 * sequence (0 for the plain recurrence) and *slice_width the V columns per
 * recurrence CTA (64 or 16). Either pointer may be NULL. varlen is nonzero for
 * a call with cu_seqlens. (A query with no counterpart on the pages; it reads
 * the device's SM count.) Returns KDA_OK, KDA_ERR_INVALID_ARG,
 * KDA_ERR_UNSUPPORTED or KDA_ERR_CUDA (no device).
 */
KDA_API kda_status_t kda_fwd_plan(int B, int T, int H, int K, int V, int num_seqs, int varlen, uint32_t flags,
                                  int *n_segments, int *slice_width);

/* Upper bound on the number of 64-token chunks over all sequences. */
KDA_API int64_t kda_max_chunks(int B, int T, int num_seqs);

/* Human-readable text of a status code (static storage, never NULL). */
KDA_API const char *kda_status_string(kda_status_t status);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device. Returns KDA_OK if no data error was recorded since the last
 * read, KDA_ERR_DEVICE_STATUS if one was (its KDA_DEVICE_* code is stored in
 * *device_code when that pointer is not NULL), or KDA_ERR_CUDA.
 */
KDA_API kda_status_t kda_get_device_status(kda_stream_t stream, int *device_code);

/*
 * Exercises the failure path of the pipeline kernels' bounded waits. One CTA
 * waits on an mbarrier that nothing arrives on, with the same bounded wait the
 * kernels use, for about limit_cycles SM clocks; it then records
 * KDA_DEVICE_WAIT_TIMEOUT in the device status word, exactly as a kernel whose
 * wait gave up does, and exits. Nothing faults or hangs and the context stays
 * usable; kda_get_device_status() then reports the code.
 * limit_cycles must be in [1, 2^32). Returns KDA_OK when the launch was
 * enqueued, KDA_ERR_INVALID_ARG for a limit out of range, KDA_ERR_CUDA.
 */
KDA_API kda_status_t kda_debug_wait_timeout(long long limit_cycles, kda_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_H_ */
