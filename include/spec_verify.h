/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) draft-then-verify acceptance
 * step of speculative decoding.  Library: libspecverify.so.
 *
 * The operation (sources named by page title and section):
 *   - "推测性拒绝采样" (speculative rejection sampling), section 技术原理与步骤:
 *     step 2, the target scores every draft prefix in one parallel pass, so
 *     its logits exist at K+1 positions; step 3, each draft token x_i is
 *     accepted when p(x_i) >= q(x_i) and otherwise with probability
 *     p(x_i)/q(x_i), and everything after the first rejection is dropped;
 *     step 4, one replacement token is drawn at the rejected position.
 *     Section 关键保证 states that the emitted tokens follow the target's own
 *     distribution exactly, which fixes the replacement law to the
 *     normalised residual max(0, p - q).
 *   - "논문 리뷰 [Speculative Contrastive Decoding]", section Speculative
 *     Decoding: when all K draft tokens are accepted the target adds token
 *     K+1 (the bonus token, drawn from p at position K).
 *   - "Garden | Blockwise Parallel Decoding", sections 3.2 and 3.5: greedy
 *     verification keeps the longest prefix on which the draft equals the
 *     target's argmax and emits the target's argmax at the first mismatch.
 *
 * Conventions shared by every entry point:
 *   - All tensors are row-major and contiguous.  Device pointers refer to
 *     memory of the current CUDA device.  The caller owns every buffer; the
 *     library allocates nothing and keeps no state between calls except a
 *     one-time per-device kernel attribute set-up on first use.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Argument errors are detected on the host before anything is launched
 *     and nothing is written then.  Errors in the data (see SPEC_DATA_*) are
 *     reported through an optional device status word, readable after the
 *     stream has been synchronised.
 *   - No entry point traps, aborts, prints, or waits on the device.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

/* A CUDA stream (the same type as cudaStream_t / CUstream). */
typedef struct CUstream_st* spec_stream_t;

/* Return codes. */
typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1,  /* bad pointer, size, dtype, mode, temperature or workspace */
  SPEC_ERR_UNSUPPORTED = 2,  /* valid request beyond the library's limits (K, V, grid) */
  SPEC_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  SPEC_ERR_SCRATCH_LIMIT = 4 /* spec_verify_static: the batch needs more scratch than
                                SPEC_STATIC_SCRATCH_BYTES */
} spec_status_t;

typedef enum {
  SPEC_MODE_SAMPLE = 0,
  SPEC_MODE_GREEDY = 1,
  SPEC_MODE_SAMPLE_EARLY_EXIT = 2  /* sampling, position 0 verified first (below) */
} spec_mode_t;
typedef enum { SPEC_DTYPE_F32 = 0, SPEC_DTYPE_BF16 = 1 } spec_dtype_t;

/* Build limits. */
#define SPEC_MAX_K 64          /* draft positions per sequence */
#define SPEC_MAX_V (1 << 22)   /* vocabulary size */

/* Device status bits (OR-ed into *device_status by the kernels).  A sequence
 * with a data error gets outputs that are in range but otherwise unspecified. */
#define SPEC_DATA_TOKEN_RANGE 1      /* a draft token outside [0, V) (clamped) */
#define SPEC_DATA_NONFINITE_LOGIT 2  /* NaN or +inf logit, or a row with no finite entry */
#define SPEC_DATA_UNIFORM_RANGE 4    /* a uniform outside [0, 1) or NaN */
/* Not a data error: one of a kernel's bounded waits -- for its own bulk
 * copies, or for work that other thread blocks of the same launch publish --
 * gave up (see spec_set_wait_limit).  The outputs of that call are then
 * unspecified and its workspace must be zero-filled again before reuse.
 * Never expected in normal use. */
#define SPEC_DEVICE_WAIT_TIMEOUT 8
#define SPEC_DATA_NONFINITE_SCORE 16 /* spec_rejection_cut: a NaN or infinite score */
/* Debug builds of the library only (compiled with -DSPEC_DEBUG, a test
 * variant): an index check on a global access failed and the access was
 * skipped instead of faulting.  A release build never sets it. */
#define SPEC_DEBUG_BOUNDS 32

/* Per-sequence boundary flags (sampling mode; written when `flags` is given).
 * They mark decisions the kernel took within 1e-6 of a threshold, where a
 * different rounding order could legitimately decide the other way. */
#define SPEC_FLAG_RATIO 1  /* |u_i - min(1, p/q)| < 1e-6 at an evaluated position i <= n */
#define SPEC_FLAG_CDF 2    /* u_K within 1e-6 (relative to the mass) of a CDF step */

/*
 * Bytes of workspace a call with these sizes needs (a multiple of 256).
 * The workspace holds per-sequence arrival counters, per-row candidates or
 * per-work-unit softmax partials (one unit is a segment of 4096 16-byte
 * vectors of a target row and its draft row), and two work counters; its
 * size grows with B, K and V * element size.  It MUST be zero-filled before its first use; every
 * call that returns SPEC_OK leaves it zero-filled again when the kernel
 * completes, so it can be reused by later calls on the same stream without
 * clearing.  One workspace serves one call at a time: calls that may overlap
 * on the GPU need separate workspaces.  Returns 0 for invalid sizes.
 */
SPEC_API size_t spec_verify_workspace_size(int B, int K, int V, int dtype, int mode);

/*
 * spec_verify -- one verify step for B independent sequences.
 *
 *   target_logits [B, K+1, V]  dtype, device.  Row (b, i) holds the target's
 *                              logits after prefix x_{<i}; row K is the bonus
 *                              position.
 *   draft_logits  [B, K, V]    dtype, device.  Row (b, i) holds the draft's
 *                              logits that x_i was sampled from.  Unused (may
 *                              be NULL) in greedy mode or when K == 0.
 *   draft_tokens  [B, K]       int32 in [0, V), device.  May be NULL if K == 0.
 *   uniforms      [B, K+1]     fp32 in [0, 1), device.  u_i (i < K) drives the
 *                              accept test of position i; u_K is the single
 *                              uniform of the replacement / bonus draw.
 *                              Unused (may be NULL) in greedy mode.
 *   B, K, V                    B >= 0 (B == 0 is a no-op), 0 <= K <= SPEC_MAX_K,
 *                              1 <= V <= SPEC_MAX_V.
 *   dtype                      SPEC_DTYPE_F32 or SPEC_DTYPE_BF16 (both logits).
 *   temperature                > 0 and finite in sampling mode: p = softmax(t/T),
 *                              q = softmax(d/T).  Ignored in greedy mode.
 *   mode                       SPEC_MODE_SAMPLE, SPEC_MODE_GREEDY or
 *                              SPEC_MODE_SAMPLE_EARLY_EXIT.
 *   accepted_len  [B]          int32 out, device: n = number of accepted draft
 *                              tokens, in [0, K].
 *   out_tokens    [B, K+1]     int32 out, device: x_0..x_{n-1}, then the
 *                              replacement (n < K) or bonus (n == K) token,
 *                              then -1 padding.
 *   workspace, workspace_bytes caller-owned device memory, at least
 *                              spec_verify_workspace_size(...) bytes, 16-byte
 *                              aligned, zero-filled before first use (above).
 *   stream                     CUDA stream the work is queued on.
 *
 * Sampling mode:  accept x_i iff u_i * q_i(x_i) < p_i(x_i); n = first rejected
 * position (K if none); at n < K the replacement is the smallest token j
 * with C_j > u_K * S, C the inclusive running sum in token order of
 * max(0, p_n - q_n) and S its total (p_n itself if S == 0); at n == K the
 * same inverse CDF is taken on p_K.
 * Early-exit sampling mode:  the same outputs as sampling mode, from a
 * schedule that stops reading a sequence's rows at its first rejection.
 * Rows whose target and draft slices fit a cluster of at most 8 CTAs (about
 * 400 KB per row at most) run one kernel in which each sequence's cluster
 * reads position i's row pair only after positions 0..i-1 were accepted,
 * and draws the replacement from the staged pair.  Longer rows read position
 * 0's row pair of every sequence first, decide position 0 and draw for each
 * sequence that rejects there; only if some sequence accepts x_0 are all rows
 * read and every sequence verified as in sampling mode.  When most sequences
 * reject their first draft token (a poor drafter) this reads about 2/(2K+1)
 * of the rows.  16-byte aligned rows with K >= 1 only; other calls run as sampling
 * mode.  p_at_draft / q_at_draft (see spec_verify_ex) are written at least
 * for positions 0..n of each sequence (the positions whose rows were read)
 * and device_status covers only the rows read.
 * Greedy mode:  g_i = argmax_j t[b, i, j] compared as fp32 values, lowest index
 * on ties; n = first i < K with x_i != g_i (K if none); the emitted token at n
 * is g_n.
 *
 * Returns SPEC_OK once the work is queued, or an error code (nothing queued).
 */
SPEC_API spec_status_t spec_verify(const void* target_logits, const void* draft_logits,
                          const int32_t* draft_tokens, const float* uniforms, int B, int K,
                          int V, int dtype, float temperature, int mode,
                          int32_t* accepted_len, int32_t* out_tokens, void* workspace,
                          size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_verify_ex -- spec_verify plus optional diagnostics (each may be NULL):
 *   p_at_draft    [B, K] fp32 out, device: p_i(x_i) for every position
 *   q_at_draft    [B, K] fp32 out, device: q_i(x_i) for every position
 *                 (both sampling mode only; left untouched in greedy mode)
 *   flags         [B] uint32 out, device: SPEC_FLAG_* bits (0 in greedy mode)
 *   device_status int32 in/out, device: the kernels OR SPEC_DATA_* bits into
 *                 it.  The caller zeroes it; it is not cleared by the library.
 */
SPEC_API spec_status_t spec_verify_ex(const void* target_logits, const void* draft_logits,
                             const int32_t* draft_tokens, const float* uniforms, int B,
                             int K, int V, int dtype, float temperature, int mode,
                             int32_t* accepted_len, int32_t* out_tokens, void* workspace,
                             size_t workspace_bytes, spec_stream_t stream,
                             float* p_at_draft, float* q_at_draft, uint32_t* flags,
                             int32_t* device_status);

/*
 * spec_verify_static -- spec_verify for callers that cannot allocate device
 * memory.  (The pages have no counterpart: this is an interface convenience.)
 *
 * Some callers cannot hand spec_verify a workspace: a host program that only
 * holds the logits and output buffers it was given by another runtime's
 * memory pool (for example an inference server that reserves all device
 * memory up front and forbids any other allocation), or a latency-critical
 * decode loop in which cudaMalloc / cudaFree are not allowed because they can
 * synchronise the device and take unbounded time.  This entry point takes the
 * same inputs and outputs as spec_verify, minus the workspace, and allocates
 * nothing: its scratch is a fixed array of SPEC_STATIC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until the process
 * exits.
 *
 *   - The batch must fit: spec_verify_workspace_size(B, K, V, dtype, mode) must
 *     not exceed SPEC_STATIC_SCRATCH_BYTES (at V = 32000 bf16, for example,
 *     B = 1024 with K = 16 or B = 4096 with K = 4 fit), else
 *     SPEC_ERR_SCRATCH_LIMIT and nothing is queued.  Other argument errors are those of spec_verify.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress, with the device current) and does the
 *     library's one-time kernel set-up; make that first call before any stream
 *     capture is started.
 *   - Every call shares the one array.  Each call clears the part it uses
 *     (cudaMemsetAsync on `stream`) before its kernel, so it does not depend
 *     on what the previous call left there; but calls that can overlap on the
 *     GPU (different streams, or different host threads) race on it and must
 *     not be issued concurrently.
 *   - Asynchronous on `stream`, like spec_verify.  No cudaMalloc, cudaFree or
 *     allocating library routine is called.
 */
#define SPEC_STATIC_SCRATCH_BYTES (1 << 20)
SPEC_API spec_status_t spec_verify_static(const void* target_logits, const void* draft_logits,
                                          const int32_t* draft_tokens, const float* uniforms,
                                          int B, int K, int V, int dtype, float temperature,
                                          int mode, int32_t* accepted_len, int32_t* out_tokens,
                                          spec_stream_t stream);

/*
 * spec_draft_sample -- the drafter's own sampling step, the one before
 * verification ("推测性拒绝采样", 技术原理与步骤 step 1; "논문 리뷰
 * [Speculative Contrastive Decoding]", Speculative Decoding: the draft model
 * samples x_i from its distribution q_i).  For each of R rows:
 *
 *   q = softmax(row / T);  x = the smallest token j with C_j > u * S, C the
 *   inclusive running sum of q in token order and S its total (the inverse
 *   CDF of spec_verify's draws).  C is summed exactly in fixed point: each
 *   16-byte vector's terms 2^((x - max)/T * log2 e) are rounded once to a
 *   multiple of 2^-40 (rows that fit a cluster's shared memory) or, for
 *   longer rows, drawn as spec_verify's bonus draw with K = 0; the two
 *   roundings can pick different tokens only when u * S lies within about
 *   1e-7 * S of a step of C.
 *
 *   logits     [R, V]  dtype, device (for example the draft's [B, K, V]
 *              logits, R = B*K).  Rows must be 16-byte aligned: V times the
 *              element size a multiple of 16, base 16-byte aligned; other
 *              rows give SPEC_ERR_UNSUPPORTED.
 *   uniforms   [R] fp32 in [0, 1), device.
 *   temperature > 0 and finite.
 *   tokens     [R] int32 out, device: x.
 *   q_at       [R] fp32 out, device, or NULL: q(x).
 *   workspace  as spec_verify's, spec_verify_workspace_size(R, 0, V, dtype,
 *              SPEC_MODE_SAMPLE) bytes, zero-filled before first use and left
 *              zero-filled.
 *   device_status  int32 in/out or NULL: SPEC_DATA_* bits, as spec_verify_ex.
 *
 * Asynchronous on `stream`; argument errors return before any launch.
 */
SPEC_API spec_status_t spec_draft_sample(const void* logits, const float* uniforms, int R, int V,
                                         int dtype, float temperature, int32_t* tokens,
                                         float* q_at, void* workspace, size_t workspace_bytes,
                                         spec_stream_t stream, int32_t* device_status);

/*
 * spec_verify_scd -- the verify step of speculative contrastive decoding
 * ("논문 리뷰 [Speculative Contrastive Decoding]", section Speculative
 * Contrastive Decoding): the amateur (the drafter) proposes x_0..x_{K-1};
 * the expert (the target) checks them against the contrastive-decoding
 * distribution P_n instead of its own p, and when all K are accepted the
 * extra token is drawn from P_n as well.  The page lost P_n's formula; this
 * library reads it as contrastive decoding's log p_e - log p_a on the
 * plausible head:
 *
 *   head_i = { j : t[b,i,j] > -inf and p_e(j) >= alpha * max p_e },
 *            p_e = softmax(t[b,i] / T), i.e. t_j >= max_j t + T ln(alpha)
 *            (taken exactly: the double max + T ln(alpha), rounded up to fp32)
 *   P_n,i(j) = exp((t[b,i,j] - a[b,i,j]) / T) / Z_i on head_i, 0 elsewhere
 *   q_i = softmax(a[b,i] / T)  (the amateur's distribution x_i was drawn from)
 *
 * and otherwise follows spec_verify's sampling mode with p replaced by P_n:
 * accept x_i iff u_i * q_i(x_i) < P_n,i(x_i); n = first rejection (K if
 * none); at n < K the token is drawn from max(0, P_n,n - q_n) (P_n,n if that
 * is zero everywhere), at n == K from P_n,K; same inverse CDF, same flags.
 *
 *   target_logits  [B, K+1, V] dtype, device: the expert's logits.
 *   amateur_logits [B, K+1, V] dtype, device: the amateur's logits; row i < K
 *                  is the distribution x_i was drawn from, row K enters only
 *                  P_n,K (the amateur's step after x_{K-1}).
 *   draft_tokens, uniforms, B, K, V, dtype, accepted_len, out_tokens,
 *   workspace, stream, p_at_draft (P_n,i(x_i)), q_at_draft, flags,
 *   device_status   as spec_verify_ex in sampling mode.  Temperature > 0.
 *   alpha          in [0, 1]: 0 keeps every token with a finite target logit,
 *                  1 only the target's argmax (then the result is greedy
 *                  verification's).
 * Rows must be 16-byte aligned (V times the element size a multiple of 16,
 * both bases 16-byte aligned): other calls return SPEC_ERR_UNSUPPORTED, as
 * do rows beyond 2^20 bf16 / 2^19 fp32 logits.  A NaN or +inf logit in either tensor, or a head
 * token whose amateur logit is -inf (an unbounded contrast), sets
 * SPEC_DATA_NONFINITE_LOGIT.  Asynchronous on `stream`.
 */
SPEC_API spec_status_t spec_verify_scd(const void* target_logits, const void* amateur_logits,
                                       const int32_t* draft_tokens, const float* uniforms, int B,
                                       int K, int V, int dtype, float temperature, double alpha,
                                       int32_t* accepted_len, int32_t* out_tokens,
                                       void* workspace, size_t workspace_bytes,
                                       spec_stream_t stream, float* p_at_draft,
                                       float* q_at_draft, uint32_t* flags,
                                       int32_t* device_status);

/*
 * spec_rejection_cut -- Speculative Rejection's cut (review "Speculative
 * Rejection", section 4.2 "算法", the speculative-rejection phase: the
 * partial responses are scored, r_cut is the alpha-quantile of the scores,
 * and the sequences scoring at least r_cut are kept for the next round).
 * For each of G prompts independently, with s its N scores sorted ascending:
 *
 *   h = alpha * (N - 1),  j = floor(h),  g = h - j,
 *   r_cut = s[j] + g * (s[min(j + 1, N - 1)] - s[j])     (IEEE double, no FMA)
 *   kept  = { k : (double)scores[k] >= r_cut }            (never empty)
 *
 * which is the usual sample quantile with linear interpolation between
 * neighbouring order statistics.
 *
 *   scores      [G, N] fp32, device, 4-byte aligned.
 *   G, N        G >= 0 (G == 0 is a no-op), N >= 1 when G > 0.
 *   alpha       in [0, 1] (the termination ratio): 0 keeps every sequence,
 *               1 keeps the best-scoring ones only.
 *   r_cut       [G] double out, device, 8-byte aligned.
 *   n_accepted  [G] int32 out, device: the number of kept sequences.
 *   accepted    [G, N] int32 out, device: row g lists the kept indices of
 *               prompt g in ascending order, then -1 up to N.
 *   device_status  int32 in/out or NULL: a prompt with a NaN or infinite
 *               score ORs SPEC_DATA_NONFINITE_SCORE into it and gets
 *               r_cut = NaN, n_accepted = 0 and a row of -1.
 *
 * No workspace.  Asynchronous on `stream`; argument errors (negative sizes,
 * N == 0 with G > 0, alpha outside [0, 1] or NaN, a NULL or misaligned
 * pointer) return SPEC_ERR_INVALID_ARG before any launch.
 */
SPEC_API spec_status_t spec_rejection_cut(const float* scores, int G, int N, double alpha,
                                          double* r_cut, int32_t* n_accepted, int32_t* accepted,
                                          spec_stream_t stream, int32_t* device_status);

/* A short, static, human-readable description of a return code. */
SPEC_API const char* spec_status_string(int status);

/*
 * spec_set_wait_limit -- bound on how long a kernel of this library waits,
 * without progress, for work that other warps or thread blocks of the same
 * launch publish (the sampling kernel for rows of at most 4096 16-byte
 * vectors decides each sequence on one thread block once the blocks that
 * streamed its rows have counted them).  Past the bound the kernel stops
 * early, ORs SPEC_DEVICE_WAIT_TIMEOUT into the device status word and leaves
 * that call's outputs unspecified, instead of waiting any longer.  The
 * limit applies to launches queued after the call, process-wide and on every
 * device.  microseconds == 0 restores the default of 2 s.  No counterpart on
 * the pages: this is the library's failure detection.  Always SPEC_OK.
 */
SPEC_API spec_status_t spec_set_wait_limit(unsigned int microseconds);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
