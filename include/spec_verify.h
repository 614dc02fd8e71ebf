/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verification library (libspecverify.so).
 *
 * One call verifies, for every sequence b of a batch, the K draft tokens
 * proposed by a draft model against the target model's logits, writes the
 * accepted prefix plus one correction (or bonus) token, and optionally the
 * per-position statistics, the logit(q_max) confidence features and the
 * online estimator's confidences.
 *
 * Sources (page title, section):
 *  [SD]  "Speculative Decoding: как черновая модель ускоряет генерацию LLM без
 *        потери качества" -- "Алгоритм на каждом шаге" (draft K tokens, one
 *        target pass, verify, append the accepted tokens plus one corrected
 *        token) and "Математика верификации" (accept x_i with probability
 *        min(1, p(x_i)/q(x_i)); on rejection draw from norm(max(0, p - q))).
 *  [AV]  "Verificación Adaptativa sin una cabeza de confianza" -- "Puntuar la
 *        Distribución" (confidence = sigmoid(omega * logit(q_max) + beta_i),
 *        K+1 parameters) and "Ajuste de los Coeficientes" (labels up to and
 *        including the first rejection).
 *  [FLy] "Training-Free Loosely Speculative Decoding: Accepting Semantically
 *        Correct Drafts Beyond Exact Match" -- 2.A.1 entropy gate, 2.A.2
 *        deferral window.
 *
 * Conventions shared by every call:
 *  - Pointers named *_logits, draft_tokens, uniforms, out_*, feature, conf,
 *    est_params, grad_out, count_out and workspace are DEVICE pointers owned
 *    by the caller (allocated e.g. through PyTorch). The library never
 *    allocates device memory and never frees what it is given.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = legacy default stream). They return after enqueueing. Host-side
 *    argument errors are reported before anything is enqueued.
 *  - Return value: SPEC_OK, or an error code below. The thread-local message
 *    of the last failure is available through spec_last_error().
 *  - Logits are row-major: target row (b, j) starts at element
 *    (b*(K+1) + j) * t_row_stride, draft row (b, i) at (b*K + i) * d_row_stride.
 *    Strides are in elements and >= V (0 means V). Every row must start on an
 *    element boundary (4-byte for fp32, 2-byte for bf16); rows starting on a
 *    16-byte boundary take the fastest path.
 *  - Logits must be finite or -inf (masked). A row whose logits are all -inf
 *    raises SPEC_ERR_BAD_ROW in the device status word (see
 *    spec_get_device_status); its outputs are then unspecified. A draft token
 *    outside [0, V) is never dereferenced: it counts as rejected and raises
 *    SPEC_ERR_BAD_TOKEN in the status word.
 *  - Outputs are deterministic: the same inputs give the same bits on every
 *    run (fixed reduction orders, no floating-point atomics).
 *  - Checked builds (compiled with SPEC_CHECKED, libspecverify_checked.so)
 *    export the same calls with the same results; their kernels also check
 *    every index they derive (work item, sequence, row, tile, draw slot,
 *    slice, token) against the buffer it addresses before the access, and
 *    on a failed check skip the access and raise SPEC_ERR_INDEX in the
 *    status word. They are for testing; the default build has no checks.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG 1   /* host-validated: nothing was enqueued   */
#define SPEC_ERR_UNSUPPORTED 2   /* shape/dtype outside the supported range */
#define SPEC_ERR_CUDA 3          /* a CUDA runtime call or launch failed    */
#define SPEC_ERR_TIMEOUT 4       /* device status: a bounded wait gave up   */
#define SPEC_ERR_BAD_ROW 5       /* device status: a row had no finite logit */
#define SPEC_ERR_BAD_TOKEN 6     /* device status: a draft token was outside [0,V) */
#define SPEC_ERR_BAD_TEMPERATURE 7 /* device status: an inverse temperature was out of range */
#define SPEC_ERR_INDEX 8         /* device status, checked builds only: an index check failed */

/* limits */
#define SPEC_MAX_B (1 << 24)     /* sequences per call                      */
#define SPEC_MAX_K 31            /* draft positions per sequence            */
#define SPEC_MAX_V (1 << 20)     /* vocabulary size                         */
#define SPEC_STATIC_SCRATCH_BYTES (16u << 20) /* scratch of spec_verify_static */
#define SPEC_MIN_INV_TEMPERATURE 1.0e-4f  /* inverse temperature range of   */
#define SPEC_MAX_INV_TEMPERATURE 1.0e4f   /* spec_verify_temperature        */

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

typedef enum {
    SPEC_STOCHASTIC = 0, /* [SD] lossless rejection rule + residual/bonus draw */
    SPEC_GREEDY = 1,     /* exact match with the target's argmax               */
    SPEC_FLY = 2         /* [FLy] entropy-gated deferral of greedy mismatches   */
} spec_mode;

typedef struct {
    int32_t B;            /* sequences, 1 .. SPEC_MAX_B                       */
    int32_t K;            /* draft positions, 1 .. SPEC_MAX_K                 */
    int32_t V;            /* vocabulary size, 2 .. SPEC_MAX_V                 */
    int32_t dtype;        /* spec_dtype of both logit tensors                 */
    int32_t mode;         /* spec_mode                                        */
    int32_t fly_window;   /* FLy: W >= 1, window of draft positions j+1..j+W  */
    float fly_theta;      /* FLy: gate threshold on normalised entropy        */
    int32_t reserved;     /* must be 0                                        */
    int64_t t_row_stride; /* elements between target rows; 0 => V             */
    int64_t d_row_stride; /* elements between draft rows; 0 => V              */
} spec_verify_params;

/*
 * Bytes of device workspace spec_verify needs for these parameters (16-byte
 * aligned allocation required). Returns 0 if the parameters are invalid.
 */
size_t spec_workspace_size(const spec_verify_params *params);

/*
 * spec_verify -- one verification pass over B sequences ([SD] steps 3-4).
 *
 * Inputs (device):
 *   target_logits [B][K+1][V]  rows 0..K-1 score the K draft tokens; row K is
 *                              the target's next-token row after all K drafts.
 *   draft_logits  [B][K][V]    the draft's rows. Required in SPEC_STOCHASTIC;
 *                              optional otherwise (NULL: no feature/conf/ratio).
 *   draft_tokens  [B][K] int32 x_i in [0, V).
 *   uniforms      [B][K+1] f32 in [0,1): u[b][i] (i < K) tests position i,
 *                              u[b][K] drives the single residual or bonus
 *                              inverse-CDF draw. Required in SPEC_STOCHASTIC,
 *                              ignored otherwise (may be NULL).
 *   est_params    [K+1] f32    (omega, beta_1..beta_K) or NULL.
 * Outputs (device):
 *   out_tokens    [B][K+1] int32  x_0..x_{n-1}, then the correction token at n,
 *                                 then -1.
 *   accepted_len  [B] int32       n in [0, K].
 *   pos_stats     [B][K+1][4] f32 or NULL: (lse of target row j, normalised
 *                                 entropy of target row j, log p(x_j) - log q(x_j),
 *                                 logit(q_max) of draft row j); the last two are
 *                                 NaN at j = K and without draft logits.
 *   feature       [B][K] f32 or NULL: logit(q_max) of every draft row,
 *                                 capped at 30 (q_max within 1e-13 of 1).
 *   conf          [B][K] f32 or NULL: sigmoid(omega*feature + beta_{i+1});
 *                                 needs est_params and draft_logits.
 * Rules:
 *   SPEC_STOCHASTIC: accept x_i iff u[b][i] < min(1, p_i(x_i)/q_i(x_i)); stop
 *     at the first rejection i and draw the correction from
 *     norm(max(0, p_i - q_i)) by inverse CDF with u[b][K] (smallest v whose
 *     running sum in ascending v exceeds u*Z); after K acceptances draw the
 *     bonus token from p_K the same way.
 *   SPEC_GREEDY: accept x_i iff x_i == argmax p_i (ties: lowest index); the
 *     correction (or bonus) is the argmax of the stop row.
 *   SPEC_FLY: a mismatch at j is rejected if h_j < fly_theta; otherwise it is
 *     accepted iff positions j+1..j+W all exist (j+W <= K-1) and all match.
 * Workspace: `workspace_bytes` >= spec_workspace_size(params); its content on
 *   entry is ignored, and it must not be shared by calls that can overlap.
 * Errors: SPEC_ERR_INVALID_ARG / SPEC_ERR_UNSUPPORTED before any launch;
 *   SPEC_ERR_CUDA if a launch fails. Device-side conditions (bad rows) land in
 *   the workspace status word.
 */
int spec_verify(const spec_verify_params *params, const void *target_logits,
                const void *draft_logits, const int32_t *draft_tokens, const float *uniforms,
                int32_t *out_tokens, int32_t *accepted_len, float *pos_stats,
                const float *est_params, float *feature, float *conf,
                void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify_static -- spec_verify without any device allocation.
 *
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory, e.g. code that runs where the allocator is
 * off limits (inside a framework that owns all device memory, a custom
 * allocator hook, or a host callback) and so cannot provide the workspace
 * spec_verify asks for. The caller still passes the inputs and outputs,
 * exactly as for spec_verify; the scratch comes from a fixed array of
 * SPEC_STATIC_SCRATCH_BYTES (16 MiB) that this library keeps in each GPU's
 * memory from the moment the library is loaded there until the process exits.
 *
 *  - Calls whose spec_workspace_size(params) exceeds that size are rejected
 *    with SPEC_ERR_UNSUPPORTED before anything is enqueued.
 *  - The call makes no cudaMalloc, cudaFree or other allocating call. Its
 *    first call on a device looks up the array's device address there
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Every call shares the one array, which keeps what the last call left
 *    in it; each call clears the parts that must start at zero. Calls that
 *    can overlap on the GPU (other streams, other threads) race on it:
 *    serialise them.
 *  - The device status word lives in that array too: read it with
 *    spec_static_device_status (not spec_get_device_status).
 * Arguments, rules and errors are those of spec_verify.
 */
int spec_verify_static(const spec_verify_params *params, const void *target_logits,
                       const void *draft_logits, const int32_t *draft_tokens, const float *uniforms,
                       int32_t *out_tokens, int32_t *accepted_len, float *pos_stats,
                       const float *est_params, float *feature, float *conf, void *stream);

/*
 * Synchronously read the device status word of the last spec_verify_static
 * call on the current device (waits for the device; allocates nothing).
 * *status_out gets SPEC_OK or the largest device-side code that call raised,
 * as for spec_get_device_status. SPEC_OK before any static call on this
 * device. Like spec_verify_static, the pages have no counterpart to it.
 */
int spec_static_device_status(int32_t *status_out);

/* Workspace bytes spec_confidence needs; 0 if the arguments are invalid. */
size_t spec_confidence_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype);

/*
 * spec_confidence -- draft-only pass ([AV] "Puntuar la Distribución"): for
 * every draft row (b, i), feature[b][i] = logit(q_max) = ln q_max - ln(1 - q_max)
 * and, if est_params and conf are given, conf[b][i] =
 * sigmoid(omega * feature + beta_{i+1}). Reads B*K*V logits once.
 * draft_logits [B][K][V] (row stride d_row_stride, 0 => V); feature [B][K]
 * required; est_params [K+1] and conf [B][K] optional (both or neither).
 */
int spec_confidence(int32_t B, int32_t K, int32_t V, int32_t dtype, const void *draft_logits,
                    int64_t d_row_stride, const float *est_params, float *feature, float *conf,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_estimator_update -- one online step of the acceptance estimator
 * ([AV] "Ajuste de los Coeficientes"). Labels: y_i = 1 for i < n_acc,
 * y_{n_acc} = 0 when n_acc < K; later positions carry no label. With
 * z = omega*f + beta_{i+1} and e = sigmoid(z) - y over the N eligible labels:
 *   g_omega = (1/N) sum e*f,  g_beta_k = (1/N) sum_{i = k-1} e,
 *   est_params -= lr * g       (no change when N = 0).
 * (The page refits by IRLS every N decoding steps; this call is one plain
 * gradient step of the mean log-loss.)
 * feature [B][K] f32, accepted_len [B] int32 in [0,K], est_params [K+1] f32
 * in/out; grad_out [K+1] f32 and count_out [K+1] int32 (N, then labels per
 * position) are optional. One CTA, fixed summation order: deterministic.
 * 1 <= K <= 1024; B >= 0.
 */
int spec_estimator_update(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                          float *est_params, float lr, float *grad_out, int32_t *count_out,
                          void *stream);

/*
 * Adaptive-verification pruning and budget ([AV] "Antecedentes", "Otras
 * Características Consideradas"). Before the target model runs, decide which
 * drafts to verify: survival[b][i] = conf[b][0] * ... * conf[b][i] (fp32
 * running product); the B*K drafts are ranked by survival (ties by the flat
 * index b*K+i, NaN last); verifying the top k is expected to emit
 * B + (sum of the top k survivals) tokens at cost draft_cost[k] +
 * verify_cost[k]; *budget = the k in 0..B*K maximising that ratio (the
 * first maximum; k with a cost that is not positive is ineligible; 0 if
 * none is eligible). Each sequence's winners are a prefix of its drafts:
 * draft_len[b] of them, the input of spec_verify_ragged.
 * Precision: the top-k sums are exact (each survival rounded to a multiple
 * of 2^-32, summed as integers); the ratio is fp32 with each step correctly
 * rounded: objective_k = (float)(B*2^32 + S_k) / (float)(draft_cost[k] +
 * verify_cost[k]) * 2^-32. The decision is therefore the same on any
 * machine that follows these steps.
 * conf [B][K] f32 in [0,1] (spec_confidence or spec_verify's conf),
 * draft_cost and verify_cost [B*K+1] f32 (caller-measured tables, k = 0..B*K),
 * draft_len [B] int32 and budget [1] int32 out; survival [B][K] f32 and
 * objective [B*K+1] f32 (-inf where ineligible) are optional outputs.
 * 1 <= B, K and B*K <= 16384 (SPEC_ERR_UNSUPPORTED beyond). One CTA;
 * bit-reproducible; asynchronous.
 */
int spec_av_budget(int32_t B, int32_t K, const float *conf, const float *draft_cost, const float *verify_cost,
                   int32_t *draft_len, int32_t *budget, float *survival, float *objective, void *stream);

/*
 * N-gram (prompt-lookup) drafting ([SD] "N-gram (prompt lookup)"; FLy's
 * "Aceleração Multinível" drafts this way): the drafts of sequence b are the
 * tokens that followed an earlier occurrence of its context's last n tokens.
 * n runs from n_max down to n_min and the longest match wins; among its
 * matches the most recent occurrence (ending last, before the context
 * does); up to K following tokens are proposed (fewer when the context
 * ends first); no match proposes none. The drafts carry no distribution, so
 * they are verified with spec_verify_ragged in greedy or FLy mode, with
 * draft_len from here.
 * ctx [B][ld] int32 (sequence b's context is ctx[b][0 .. len[b]-1], len
 * clamped to [0, ld]), draft_tokens [B][K] int32 out (-1 past the drafts),
 * draft_len [B] int32 out. 1 <= n_min <= n_max, K >= 1. One warp per
 * sequence, integer work: exact. Asynchronous on `stream`.
 */
int spec_ngram_draft(int32_t B, int32_t ld, const int32_t *ctx, const int32_t *len, int32_t n_min, int32_t n_max,
                     int32_t K, int32_t *draft_tokens, int32_t *draft_len, void *stream);

/*
 * spec_verify for a pruned batch: sequence b submitted only its first
 * draft_len[b] drafts for verification ([AV]: a subset of the drafts is
 * verified; the target ran with variable-length sequences). draft_len [B]
 * int32 on the device, each clamped to [0, K]. Sequence b verifies drafts
 * 0..kb-1 against target rows 0..kb (kb = draft_len[b]); after kb acceptances
 * the bonus token comes from target row kb; the final draw still uses
 * uniforms[b][K]; FLy's window must fit inside kb. Rows never verified are
 * not read: their pos_stats, feature and conf entries are NaN and their
 * out_tokens -1. Layouts, workspace and status codes are spec_verify's (the
 * logit tensors keep their [B][K+1][V] / [B][K][V] layout).
 */
int spec_verify_ragged(const spec_verify_params *params, const void *target_logits, const void *draft_logits,
                       const int32_t *draft_tokens, const int32_t *draft_len, const float *uniforms,
                       int32_t *out_tokens, int32_t *accepted_len, float *pos_stats, const float *est_params,
                       float *feature, float *conf, void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify at a sampling temperature ([AV] "Benchmarks": the serving
 * setting samples at a temperature; [SD] "Математика верификации": the rule
 * is lossless for whatever distributions the two models sample from).
 * inv_temperature [B] f32 on the device holds s_b = 1/T_b per sequence, in
 * [SPEC_MIN_INV_TEMPERATURE, SPEC_MAX_INV_TEMPERATURE]. Both models' rows of
 * sequence b are processed as p = softmax(s_b z), q = softmax(s_b y) before
 * every use: the acceptance ratio, the residual and bonus draws, the FLy
 * entropy, logit(q_max) and pos_stats' lse and log-ratio all read the
 * processed distributions (argmax decisions do not change). The caller draws
 * the drafts from the processed q. draft_len may be NULL (all K verified) or
 * as for spec_verify_ragged. A value outside the range (or NaN) runs that
 * sequence at s = 1 and sets SPEC_ERR_BAD_TEMPERATURE in the status word.
 * Everything else is spec_verify's. Exponents are formed difference first,
 * (z - M) s log2e, so that accuracy does not degrade with |s z|; at s = 1
 * results therefore agree with spec_verify's to a few fp32 roundings, not
 * bit for bit. An inverse temperature 2^k on z gives the bits of s = 1 on
 * 2^k z.
 */
int spec_verify_temperature(const spec_verify_params *params, const void *target_logits,
                            const void *draft_logits, const int32_t *draft_tokens, const int32_t *draft_len,
                            const float *inv_temperature, const float *uniforms, int32_t *out_tokens,
                            int32_t *accepted_len, float *pos_stats, const float *est_params, float *feature,
                            float *conf, void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify at a sampling top-p, after an optional temperature ([AV]
 * "Benchmarks": the serving setting samples with top-p 0.95; [SD]
 * "Математика верификации": the rule is lossless for the distributions the
 * models sample from). Every row (target and draft) is processed as
 * p = softmax(s_b z) restricted to its nucleus and renormalised: the nucleus
 * is every token whose logit is at least z*, the largest logit value whose
 * tokens (logit >= z*) hold at least top_p of the row's mass; tokens tied
 * at z* are all kept. The acceptance ratio, residual and bonus draws, FLy
 * entropy, logit(q_max) and pos_stats read the processed rows; a token
 * outside a nucleus has probability 0 there (its log-ratio is -inf, or +inf
 * when only the draft's nucleus excludes it). The caller draws the drafts
 * from the processed q.
 *   top_p            in (0, 1]; 1 is spec_verify_temperature (or spec_verify
 *                    when inv_temperature is NULL).
 *   inv_temperature  [B] f32 or NULL (s = 1); as for spec_verify_temperature.
 *   draft_len        [B] int32 or NULL; as for spec_verify_ragged.
 * Cost: a nucleus pass precedes the verification launch. A thread-block
 * cluster holds each row in shared memory for the threshold search: one HBM
 * read per row, for 16-byte aligned rows of up to 256 KB per 8 CTAs. Other
 * rows take one CTA per row, re-read from L2. Workspace, layouts and status
 * codes are spec_verify's. Errors: SPEC_ERR_INVALID_ARG for top_p outside
 * (0, 1].
 */
int spec_verify_top_p(const spec_verify_params *params, const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, const int32_t *draft_len, const float *inv_temperature,
                      float top_p, const float *uniforms, int32_t *out_tokens, int32_t *accepted_len,
                      float *pos_stats, const float *est_params, float *feature, float *conf, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * spec_estimator_update and spec_irls_accumulate for a pruned batch: only
 * verified drafts carry labels, so with kb = draft_len[b] the label at
 * position n_acc (y = 0) exists only when n_acc < kb, and positions >= kb
 * carry none. accepted_len[b] must lie in [0, kb].
 */
int spec_estimator_update_ragged(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                                 const int32_t *draft_len, float *est_params, float lr, float *grad_out,
                                 int32_t *count_out, void *stream);
int spec_irls_accumulate_ragged(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                                const int32_t *draft_len, const float *est_params, void *state, void *stream);

/*
 * IRLS refit of the acceptance estimator ([AV] "Ajuste de los Coeficientes").
 * The coefficients est_params = (omega, beta_1..beta_K) stay fixed over a
 * round of decoding steps; each step adds the gradient g and Hessian H of
 * the summed log-loss of its eligible labels (labelled as for
 * spec_estimator_update) to a device-resident round state; after the
 * round's last step the refit solves H d = g and moves every coefficient by
 * d damped by n / (n + damping), n being the labels behind it (the slope:
 * all of the round's labels; beta_k: the labels at draft position k).
 * The pages leave the round length N and the constant c open: the caller
 * chooses them by when it calls spec_irls_refit and with which damping.
 *
 * State: spec_irls_state_size(K) bytes of caller-owned device memory, 8-byte
 * aligned, of 4K+3 doubles: g[0..K] (g[0] the slope, g[1+i] draft position
 * i), H_ww, H_wb[0..K-1], H_bb[0..K-1], n[0..K] (n[0] all labels, n[1+i]
 * labels at position i). H is an arrow matrix (one label touches the slope
 * and one intercept), so these entries are all of it. spec_irls_reset
 * zeroes it; spec_irls_refit zeroes it after using it.
 *
 * Refit readings (the pages are silent): coefficients without labels keep
 * their value; if after eliminating the intercepts the slope's pivot is at
 * most 1e-12 of H_ww (the round does not determine the slope), the slope is
 * held and the intercepts solve with it fixed. A round without labels
 * changes nothing. step_out [K+1] doubles (optional) receives the applied
 * step (params -= step).
 *
 * feature [B][K] f32 and accepted_len [B] int32 in [0,K] as produced by
 * spec_verify; est_params [K+1] f32 (read by accumulate, updated by refit).
 * Precision: each label's sigmoid terms are fp32; every sum and the solve
 * are fp64. 1 <= K <= 1024; B >= 0. One CTA each, fixed summation order:
 * the results are bit-reproducible. Asynchronous on `stream`; the status
 * codes are those of spec_verify.
 */
size_t spec_irls_state_size(int32_t K);
int spec_irls_reset(int32_t K, void *state, void *stream);
int spec_irls_accumulate(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                         const float *est_params, void *state, void *stream);
int spec_irls_refit(int32_t K, void *state, float *est_params, double damping, double *step_out,
                    void *stream);

/*
 * Synchronously read the device status word of a workspace last used by
 * spec_verify or spec_confidence (waits for the device). *status_out gets
 * SPEC_OK or the largest device-side code raised (SPEC_ERR_TIMEOUT,
 * SPEC_ERR_BAD_ROW, SPEC_ERR_BAD_TOKEN). For tests and debugging.
 */
int spec_get_device_status(const void *workspace, int32_t *status_out);

/*
 * Testing hook for the bounded waits (no counterpart on the pages). A warp of
 * the verification kernel whose stream work is done waits for the draw of
 * the residual unit it claimed; it polls at most `polls` times (default
 * 2^20, well under a second) before it raises SPEC_ERR_TIMEOUT in the status
 * word and leaves that work undone. 0 makes every such wait give up at once,
 * so that a test can see the timeout path without a hang: the outputs of
 * the draw are then unspecified. The setting applies to launches enqueued
 * after the call, from any thread; returns the previous setting.
 */
uint32_t spec_debug_set_wait_limit(uint32_t polls);

/* Message of the calling thread's last failure ("" if none). */
const char *spec_last_error(void);

/* Library version string. */
const char *spec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
