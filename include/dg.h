/*
 * dg.h -- C ABI of libdg, the GB300 (sm_103a) entropy-bounded denoising step of a
 * block-diffusion language model with fixed-length canvases.
 *
 * Sources (web pages, cited by title and section):
 *   [DG]  "DiffusionGemma: vLLM이 네이티브로 지원하는 최초의 디퓨전 언어 모델(dLLM)"
 *         (discuss.pytorch.kr):
 *           - "엔트로피 기반 디노이징" (entropy-based denoising): every step resamples all
 *             canvas positions, keeps the confident ones and renoises the rest; the
 *             entropy H(p) = -sum_i p_i log p_i; the entropy-bound acceptance rule; the
 *             convergence rule (argmax unchanged for several steps AND mean entropy below
 *             a threshold, or the step cap), after which the argmax canvas is committed.
 *           - "자기 조건화" (self-conditioning): the previous step's softmax becomes a
 *             probability-weighted mean of token embeddings, goes through a small gated
 *             MLP and is added to the next pass's canvas embeddings; zero for the encoder
 *             prefill and commit passes.
 *           - "DiffusionGemmaModelState와 DiffusionSampler": the Prefill case (random
 *             canvas), the Denoise case (logits / T, Gumbel-max candidates
 *             argmax(logits / T + g), entropy-bound acceptance, renoise, argmax canvas,
 *             convergence check) and the per-request state kept in pre-allocated GPU
 *             tensors updated in place.
 *   [SPR] "답은 한 번 읽는데 모델은 왜 두 번 돌까? DiffusionGemma의 실행 경로 합치기":
 *         read-only requests take a single denoising pass and only read probabilities
 *         (diffusion_read_only with diffusion_max_steps = 1).
 *   [PHX] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 *         SC'11 (Philox-4x32, 10 rounds).
 *
 * Conventions for every entry point:
 *   - Pointers marked (device) are device pointers owned by the caller; the library never
 *     allocates, frees or keeps them.  Pointers marked (host) are read during the call.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *     and is asynchronous: outputs are valid once the stream has reached the call.
 *   - The return value reports host-side validation and launch errors only.  On a
 *     validation error nothing is launched and no output is touched.  Problems found in
 *     device data (NaN / +inf logits, all -inf rows, an expired bounded wait) set bits in
 *     a device status word, read with dg_get_device_status().  Kernels never trap.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Layouts are row-major.  "[n][L]" means canvas-major, position-minor, contiguous.
 *   - Kernels are compiled for sm_103a only; on another device every launch returns
 *     DG_ERR_CUDA.
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported entry points (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define DG_API __attribute__((visibility("default")))
#else
#define DG_API
#endif

typedef struct CUstream_st* dg_stream_t; /* same type as cudaStream_t */

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = -1, /* null pointer, size out of range, bad dtype            */
    DG_ERR_ALIGNMENT = -2,   /* a pointer or row stride breaks the alignment rules    */
    DG_ERR_WORKSPACE = -3,   /* workspace null or smaller than *_workspace_bytes()    */
    DG_ERR_UNSUPPORTED = -4, /* shape outside what the kernels handle (see each call) */
    DG_ERR_CUDA = -5         /* a CUDA runtime call or launch failed                  */
} dg_status;

typedef enum { DG_BF16 = 0, DG_FP32 = 1 } dg_dtype;

/* Per-canvas flags. */
enum {
    DG_ACTIVE = 1u,    /* the canvas takes part in this step; clear = already converged:
                          its logits are never read and none of its outputs is written  */
    DG_READ_ONLY = 2u, /* single-pass read [SPR]: statistics only (entropy, lse, argmax);
                          nothing accepted, canvas unchanged, converged = 1              */
    DG_SELF_COND = 4u, /* compute the self-conditioning feedback for this canvas [DG]    */
    DG_SAMPLE_ALL = 8u /* draw the Gumbel-max sample at every position; clear = only at
                          the accepted positions, the only ones whose sample is kept      */
};

/* Bits of the device status word. */
enum {
    DG_DEV_NAN_INF_ROW = 1u, /* a row held NaN or +inf logits; its outputs are unspecified */
    DG_DEV_EMPTY_ROW = 2u,   /* a row was all -inf; its outputs are unspecified           */
    DG_DEV_TIMEOUT = 4u,     /* a bounded wait inside a kernel expired; outputs of that
                                launch are unspecified and the context stays usable       */
    DG_DEV_BAD_PARAM = 8u    /* a per-canvas parameter was out of range (T <= 0, k < 1,
                                max_steps < 1, min_accept outside 0..L); that canvas is
                                skipped                                                   */
};

/* Per-canvas parameters, one 36-byte record per canvas, in device memory.
 * The Philox key for a canvas is (lo32(seed), request_id); the counter is
 * (block, position, step, stream | bits 32..55 of seed << 8) with stream 0 = Gumbel noise,
 * 1 = renoise tokens, 2 = canvas initialisation [PHX]. */
typedef struct {
    float temperature;   /* T > 0: logits are scaled by 1/T [DG Denoise case]            */
    float beta;          /* entropy budget in nats [DG entropy-bound rule]                */
    float tau;           /* mean-entropy threshold in nats [DG convergence rule]          */
    int32_t k;           /* consecutive unchanged argmax steps required, >= 1             */
    int32_t max_steps;   /* step cap S >= 1: converged once step + 1 >= S                 */
    int32_t min_accept;  /* positions accepted even when the budget allows none (0..L)    */
    int32_t step;        /* 0-based index of this denoising step for the canvas           */
    uint32_t request_id; /* second Philox key word                                        */
    uint32_t flags;      /* DG_ACTIVE | DG_READ_ONLY | DG_SELF_COND | DG_SAMPLE_ALL        */
} dg_canvas_params;

/* ------------------------------------------------------------------------------------ */
/* Denoise step [DG "엔트로피 기반 디노이징", "DiffusionGemmaModelState와 DiffusionSampler"]. */
/* ------------------------------------------------------------------------------------ */

/* Workspace needed by dg_denoise_step: the list of accepted positions that the deferred
 * sampling launch works through (256 bytes + 24 bytes per position, rounded up to 256). */
DG_API size_t dg_denoise_workspace_bytes(int64_t n_canvas, int32_t L, int64_t V, dg_dtype dtype);

/* One denoising step for n_canvas canvases of L positions over a vocabulary of V.
 *
 * For each position of each DG_ACTIVE canvas, with y = logits / T:
 *   entropy = H(softmax(y)) = -sum p log p (nats), lse = log sum exp(y),
 *   argmax  = smallest v with logits[v] = max (the raw logits),
 *   sample  = smallest v maximising y_v + g_v, g_v = -log(-log u_v) Gumbel noise from
 *             Philox stream 0 with block = v / 4, word = v % 4, and
 *             u = (floor(w / 2^9) + 1/2) / 2^23.
 * Then per canvas: positions are ordered by (entropy, position) ascending and accepted
 * while the running sum of their entropies stays <= beta (at least min_accept, at most L);
 * accepted positions take their sample, the others a uniform token over [0, V) from
 * Philox stream 1 (block 0, token = floor((w0 << 32 | w1) * V / 2^64)).  Convergence:
 * stable_count becomes stable_count + 1 when the whole argmax canvas equals prev_argmax,
 * else 0; the canvas converges when (stable_count >= k and mean entropy < tau) or
 * step + 1 >= max_steps; prev_argmax is then overwritten with argmax.  DG_READ_ONLY canvases compute entropy,
 * lse and argmax only (sample = -1, accept_mask = 0, canvas unchanged, converged = 1).
 *
 * Where the sample is drawn: a rejected position's sample is replaced by its renoise token
 * in the same step, so by default the sample is drawn only after the acceptance, at the
 * accepted positions (a second read of those rows); sample = -1 at the rejected ones.  The
 * canvas, accept mask and every other output are the same either way.  With DG_SAMPLE_ALL
 * set on a canvas, every position of it draws its sample in the statistics pass (sample
 * defined everywhere).  The launches are: statistics (+ samples of DG_SAMPLE_ALL canvases),
 * acceptance / renoise / convergence (which lists the accepted positions of the other
 * canvases in the workspace), then the samples of the listed positions (16 KB of a row per
 * warp; results do not depend on which warp finishes first).
 *
 *   logits        (device) [n_canvas][L][ld] of dtype; 16-byte aligned; ld >= V and
 *                 ld * sizeof(dtype) a multiple of 16.  Columns V..ld-1 are never read.
 *   params        (device) [n_canvas] dg_canvas_params.
 *   seed          Philox seed (low 32 bits = key word 0, bits 32..55 in the counter).
 *   canvas        (device, in/out) [n_canvas][L] int32: the next canvas, written in place.
 *   prev_argmax   (device, in/out) [n_canvas][L] int32: previous argmax canvas; -1 = none.
 *   stable_count  (device, in/out) [n_canvas] int32.
 *   accept_mask   (device, out) [n_canvas][L] uint8 (1 = accepted).
 *   argmax, sample(device, out) [n_canvas][L] int32 (sample: -1 where not drawn, see above).
 *   entropy, lse  (device, out) [n_canvas][L] float.
 *   converged     (device, out) [n_canvas] uint8.
 *   mean_entropy  (device, out, may be NULL) [n_canvas] float.
 *   n_accept      (device, out, may be NULL) [n_canvas] int32.
 *   workspace     (device) at least dg_denoise_workspace_bytes() bytes, 8-byte aligned;
 *                 scratch owned by the call until the stream passes it (no initial
 *                 contents needed); calls that overlap on the GPU need their own.
 * Limits: 1 <= L <= 1024, 2 <= V < 2^31, 0 <= n_canvas <= 65535 (0 launches nothing), and
 * V * sizeof(dtype) < 2^31 bytes (else DG_ERR_UNSUPPORTED).
 * Errors: DG_ERR_INVALID_ARG (null required pointer, sizes), DG_ERR_ALIGNMENT,
 * DG_ERR_WORKSPACE (workspace null or too small), DG_ERR_UNSUPPORTED, DG_ERR_CUDA. */
DG_API dg_status dg_denoise_step(const void* logits, dg_dtype dtype, int64_t ld,
                          int64_t n_canvas, int32_t L, int64_t V,
                          const dg_canvas_params* params, uint64_t seed,
                          int32_t* canvas, int32_t* prev_argmax, int32_t* stable_count,
                          uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                          float* entropy, float* lse, uint8_t* converged,
                          float* mean_entropy, int32_t* n_accept,
                          void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* dg_denoise_step in two calls, so that the samples can run on another stream (e.g. beside
 * the self-conditioning GEMMs, which do not read them):
 *   dg_denoise_stats:   statistics, acceptance, renoise of the rejected positions and
 *                       convergence; lists the accepted positions of canvases without
 *                       DG_SAMPLE_ALL in the workspace (their sample and canvas entries are
 *                       written by dg_denoise_samples);
 *   dg_denoise_samples: the Gumbel-max samples of the listed positions, written to sample
 *                       and canvas.  It launches at most one CTA per SM (of 96 threads and
 *                       at most 80 registers, no shared memory), so that it can share SMs
 *                       with a GEMM running on another stream (a P.E CTA of 448 threads x
 *                       128 registers leaves room for it).
 * dg_denoise_samples must follow dg_denoise_stats of the same step (an event on the stats'
 * stream when it runs on another stream), with the same logits, params, seed, sizes and
 * workspace, and complete before the canvas or the workspace is used again (by the caller or
 * the next step).  Arguments, limits and errors are those of dg_denoise_step; together the
 * two calls produce exactly its outputs. */
DG_API dg_status dg_denoise_stats(const void* logits, dg_dtype dtype, int64_t ld,
                                  int64_t n_canvas, int32_t L, int64_t V,
                                  const dg_canvas_params* params, uint64_t seed,
                                  int32_t* canvas, int32_t* prev_argmax, int32_t* stable_count,
                                  uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                                  float* entropy, float* lse, uint8_t* converged,
                                  float* mean_entropy, int32_t* n_accept,
                                  void* workspace, size_t workspace_bytes, dg_stream_t stream);
DG_API dg_status dg_denoise_samples(const void* logits, dg_dtype dtype, int64_t ld,
                                    int64_t n_canvas, int32_t L, int64_t V,
                                    const dg_canvas_params* params, uint64_t seed,
                                    int32_t* canvas, int32_t* sample,
                                    void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* dg_denoise_step with the single-pass-read gather fused into the statistics pass [SPR,
 * "답의 내용은 몰라도 답을 담을 자리는 안다": one pass over a read-only request's logits
 * returns the probabilities of its fixed answer tokens].  Besides every output of
 * dg_denoise_step, for every position of every DG_ACTIVE canvas and every slot k < C:
 *   probs[c][i][k] = exp(logits[c][i][tok] / T - lse[c][i]),  tok = choices[c][i][k],
 * with the lse this call writes; the CTA that streams the row gathers its C logits as soon as
 * its lse is known, so the logits are not read a second time.  The values are those of
 * dg_choice_probs on this call's lse (bit for bit).  A slot with a token outside [0, V)
 * gives 0 (use -1 for unused slots); inactive canvases leave probs untouched.  Read-only
 * canvases (DG_READ_ONLY) are the intended users, but every active canvas is served.
 *   choices (device) [n_canvas][L][C] int32.
 *   probs   (device, out) [n_canvas][L][C] float.
 * Other arguments, limits and errors are those of dg_denoise_step; in addition
 * DG_ERR_INVALID_ARG for C outside [1, 1024] or null choices / probs. */
DG_API dg_status dg_denoise_step_choices(const void* logits, dg_dtype dtype, int64_t ld,
                                         int64_t n_canvas, int32_t L, int64_t V,
                                         const dg_canvas_params* params, uint64_t seed,
                                         int32_t* canvas, int32_t* prev_argmax, int32_t* stable_count,
                                         uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                                         float* entropy, float* lse, uint8_t* converged,
                                         float* mean_entropy, int32_t* n_accept,
                                         const int32_t* choices, int32_t C, float* probs,
                                         void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* dg_denoise_stats in two calls, so that the acceptance (and then dg_denoise_samples) can run
 * on another stream while the self-conditioning feedback, which needs only lse, starts:
 *   dg_denoise_row_stats: per-position entropy, lse, argmax (and the samples of DG_SAMPLE_ALL
 *                         canvases; -1 elsewhere), each row's maximum recorded in the
 *                         workspace and the workspace's list cleared;
 *   dg_denoise_accept:    acceptance, renoise, convergence and the list of accepted positions
 *                         (exactly the second half of dg_denoise_stats, on the outputs of
 *                         dg_denoise_row_stats and the same workspace).  The next launch on its
 *                         stream starts only when it completes; up to 256 positions its CTAs
 *                         use 256 threads and at most 32 registers, so that each fits on an
 *                         SM beside a feedback GEMM CTA.
 * In order (dg_denoise_row_stats, dg_denoise_accept, dg_denoise_samples, with the same
 * logits, params, seed, sizes and workspace) they produce exactly dg_denoise_step's outputs.
 * Arguments, limits and errors are those of dg_denoise_step (dg_denoise_accept checks the
 * workspace size as for bf16 logits, which is the same for every dtype). */
DG_API dg_status dg_denoise_row_stats(const void* logits, dg_dtype dtype, int64_t ld,
                                      int64_t n_canvas, int32_t L, int64_t V,
                                      const dg_canvas_params* params, uint64_t seed,
                                      int32_t* argmax, int32_t* sample, float* entropy, float* lse,
                                      void* workspace, size_t workspace_bytes, dg_stream_t stream);
DG_API dg_status dg_denoise_accept(const float* entropy, const int32_t* sample, const int32_t* argmax,
                                   int64_t n_canvas, int32_t L, int64_t V,
                                   const dg_canvas_params* params, uint64_t seed,
                                   int32_t* canvas, int32_t* prev_argmax, int32_t* stable_count,
                                   uint8_t* accept_mask, uint8_t* converged,
                                   float* mean_entropy, int32_t* n_accept,
                                   void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* The per-canvas half of the step (acceptance, renoise, convergence) on caller-given
 * per-position entropy, sample and argmax, all (device) [n_canvas][L].  Same semantics and
 * outputs as dg_denoise_step, except that every accepted position takes the given sample
 * (DG_SAMPLE_ALL plays no part); used to test the acceptance rule on chosen entropies. */
DG_API dg_status dg_accept_from_entropy(const float* entropy, const int32_t* sample,
                                 const int32_t* argmax, int64_t n_canvas, int32_t L, int64_t V,
                                 const dg_canvas_params* params, uint64_t seed,
                                 int32_t* canvas, int32_t* prev_argmax, int32_t* stable_count,
                                 uint8_t* accept_mask, uint8_t* converged,
                                 float* mean_entropy, int32_t* n_accept, dg_stream_t stream);

/* Prefill case [DG "DiffusionGemmaModelState와 DiffusionSampler"]: fill every DG_ACTIVE
 * canvas with uniform tokens over [0, V) from Philox stream 2 (block 0, counter step =
 * params.step).  canvas (device, out) [n_canvas][L] int32.  Same limits as above. */
DG_API dg_status dg_canvas_init(int32_t* canvas, int64_t n_canvas, int32_t L, int64_t V,
                         const dg_canvas_params* params, uint64_t seed, dg_stream_t stream);

/* Between steps of a loop: for every canvas, clear DG_ACTIVE when converged[c] is 1 and
 * advance step by one otherwise (the canvas then commits its argmax [DG convergence
 * rule]).  params (device, in/out) [n_canvas]; converged (device) [n_canvas]. */
DG_API dg_status dg_advance_params(dg_canvas_params* params, const uint8_t* converged,
                            int64_t n_canvas, dg_stream_t stream);

/* ------------------------------------------------------------------------------------ */
/* LM head fused with the step's statistics.  The logits the denoise step reads are the   */
/* model's output over the canvas [DG "엔트로피 기반 디노이징"]; the pages do not describe  */
/* the output layer, and the reading taken is a plain linear map of the last hidden        */
/* states, logits = bf16(hidden . W_lm^T), no bias, no soft-capping (W_lm is the input    */
/* embedding table when the model ties them).  Computed on the tensor cores (tcgen05,      */
/* bf16 operands, fp32 accumulation, one rounding to bf16 per logit); the statistics are   */
/* taken from the stored bf16 logits in the GEMM's epilogue, so the logits are not read    */
/* back for them.                                                                          */
/* ------------------------------------------------------------------------------------ */

/* Workspace for dg_lm_head_logits / dg_lm_head_denoise_step (bytes): the deferred-sampling
 * list of dg_denoise_workspace_bytes, the list of active canvases, and 20 bytes per position
 * and 256 columns of V (each row's softmax state per tile). */
DG_API size_t dg_lm_head_workspace_bytes(int64_t n_canvas, int32_t L, int64_t V);

/* logits = bf16(hidden . W_lm^T) for every position of every DG_ACTIVE canvas; the rows of
 * other canvases are not written.
 *   hidden  (device) [n_canvas][L][ldh] bf16: last hidden states; ldh >= d, ldh % 8 == 0.
 *   W_lm    (device) [V][ldw] bf16: output projection (row v = token v); ldw >= d, % 8 == 0.
 *   logits  (device, out) [n_canvas][L][ld] bf16; ld >= V, ld % 8 == 0.  Columns V..ld-1
 *           are not written.
 *   params  (device) [n_canvas]: only DG_ACTIVE is read.
 *   workspace (device) >= dg_lm_head_workspace_bytes(), 16-byte aligned, no initial contents.
 * All device pointers 16-byte aligned.  Limits: 8 <= d <= 65536, d % 8 == 0, V < 2^30;
 * n_canvas and L as dg_denoise_step.  Errors: DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT,
 * DG_ERR_WORKSPACE, DG_ERR_CUDA.  Enqueues 2 kernels. */
DG_API dg_status dg_lm_head_logits(const uint16_t* hidden, int64_t ldh, const uint16_t* W_lm,
                                   int64_t ldw, int64_t n_canvas, int32_t L, int64_t V, int32_t d,
                                   const dg_canvas_params* params, uint16_t* logits, int64_t ld,
                                   void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* dg_lm_head_logits, then one denoising step on those logits: the outputs of
 * dg_denoise_step (same meaning, same arguments after params) for the logits it stores,
 * which the self-conditioning calls can then read with the lse written here.  Every
 * canvas is sampled at its accepted positions only (DG_SAMPLE_ALL has no effect: sample
 * is -1 at the other positions).  Launches: active-canvas list, the LM-head GEMM with the
 * statistics epilogue, a merge of the per-tile states (fixed order: results do not depend
 * on timing), acceptance / renoise / convergence, the samples of the accepted positions.
 * Same limits and errors as dg_lm_head_logits and dg_denoise_step. */
DG_API dg_status dg_lm_head_denoise_step(const uint16_t* hidden, int64_t ldh, const uint16_t* W_lm,
                                         int64_t ldw, int64_t n_canvas, int32_t L, int64_t V,
                                         int32_t d, const dg_canvas_params* params, uint64_t seed,
                                         uint16_t* logits, int64_t ld, int32_t* canvas,
                                         int32_t* prev_argmax, int32_t* stable_count,
                                         uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                                         float* entropy, float* lse, uint8_t* converged,
                                         float* mean_entropy, int32_t* n_accept,
                                         void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* ------------------------------------------------------------------------------------ */
/* Attention with per-sequence causality [DG "시퀀스별로 동적으로 바뀌는 인과 어텐션",       */
/* "슬라이딩 윈도우 어텐션도 대칭으로"]: one batch mixes causal requests (prefill / commit   */
/* passes) and bidirectional ones (a denoising canvas, which sees its context and the whole */
/* canvas); key tiles that hold no allowed key are skipped (neither loaded nor multiplied). */
/* ------------------------------------------------------------------------------------ */

/* o[i][h] = softmax over the allowed keys j of (scale * q[i][h] . k[j][h']) applied to v,
 * h' = h / (Hq / Hkv), for every query of n_seq sequences.  Sequence s owns queries
 * cu_q[s] .. cu_q[s+1]-1 and keys cu_kv[s] .. cu_kv[s+1]-1; its queries are its last
 * q_len = cu_q[s+1] - cu_q[s] tokens, so query i sits at position kv_len - q_len + i.  Key j
 * is allowed when j < kv_len and, for causal[s] != 0, j <= position; with window >= 0 also
 * j >= position - window and, for a bidirectional sequence, j <= position + window.
 *   q    (device) [total_q][Hq][D] bf16;  k, v (device) [total_kv][Hkv][D] bf16.
 *   o    (device, out) [total_q][Hq][D] bf16.
 *   lse  (device, out, may be NULL) [total_q][Hq] float: log sum exp of the allowed scores.
 *   cu_q, cu_kv (device) [n_seq + 1] int32 offsets (non-decreasing); causal (device) [n_seq].
 *   max_q_len: at least every sequence's q_len (a smaller one leaves the queries past it out
 *   and raises DG_DEV_BAD_PARAM); a sequence with q_len > kv_len or offsets outside
 *   [0, total_q] / [0, total_kv] raises DG_DEV_BAD_PARAM and is skipped (its rows of o are not
 *   written).
 *   workspace (device) >= dg_attention_workspace_bytes(n_seq, max_q_len), 16-byte aligned,
 *   no initial contents: the list of (sequence, query tile) items, longest first.
 * D must be 64, 128 or 256 (else DG_ERR_UNSUPPORTED); Hq a multiple of Hkv; window >= -1 (-1: none);
 * total_q, total_kv < 2^31; q, k, v, o 16-byte aligned.  Computed on the tensor cores
 * (tcgen05, bf16 operands, fp32 accumulation and softmax, one pass) by persistent CTAs (two
 * per SM for D = 64 and 128, one for D = 256) that take the listed items in turn.  Two kernel launches (the list, the attention). */
DG_API size_t dg_attention_workspace_bytes(int32_t n_seq, int32_t max_q_len);
DG_API dg_status dg_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                              float* lse, const int32_t* cu_q, const int32_t* cu_kv,
                              const uint8_t* causal, int32_t n_seq, int32_t max_q_len,
                              int64_t total_q, int64_t total_kv, int32_t Hq, int32_t Hkv, int32_t D,
                              int32_t window, float scale, void* workspace, size_t workspace_bytes,
                              dg_stream_t stream);

/* ------------------------------------------------------------------------------------ */
/* Self-conditioning [DG "자기 조건화"]:                                                  */
/*   pe    = P . E,  P = softmax(logits / T) per position, E the token embedding table;  */
/*   delta = W_down (gelu_tanh(W_gate pe) * (W_up pe)), no bias (gated MLP).            */
/* Computed on the tensor cores (tcgen05, bf16 operands, fp32 accumulation); P is formed */
/* tile by tile in shared memory from the logits and the step's lse, never in HBM.      */
/* ------------------------------------------------------------------------------------ */

/* Workspace for dg_self_cond_logits with these sizes (bytes, 256-byte aligned use). */
DG_API size_t dg_self_cond_workspace_bytes(int64_t n_canvas, int32_t L, int32_t d, int32_t h);

/* delta_emb for every position of every canvas with DG_ACTIVE and DG_SELF_COND set, not
 * DG_READ_ONLY and not converged in this step; all other rows of delta_emb are set to 0
 * (the feedback is zero for the prefill and commit passes [DG "자기 조건화"]).
 *   logits    (device) [n_canvas][L][ld] as in dg_denoise_step.
 *   lse       (device) [n_canvas][L] float: the lse output of dg_denoise_step for these
 *             logits and parameters.
 *   params    (device) [n_canvas]; converged (device) [n_canvas] uint8 (may be NULL =
 *             none converged).
 *   E         (device) bf16 [V][d] token embeddings; W_gate, W_up (device) bf16 [h][d];
 *             W_down (device) bf16 [d][h] (row = output unit).  All 16-byte aligned.
 *   delta_emb (device, out) bf16 [n_canvas][L][d].
 * Limits: d and h multiples of 8 in [8, 65536]; L <= 1024; V as in dg_denoise_step.
 * Errors: DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT, DG_ERR_WORKSPACE, DG_ERR_CUDA. */
DG_API dg_status dg_self_cond_logits(const void* logits, dg_dtype dtype, int64_t ld, const float* lse,
                              const dg_canvas_params* params, const uint8_t* converged,
                              int64_t n_canvas, int32_t L, int64_t V, int32_t d, int32_t h,
                              const uint16_t* E, const uint16_t* W_gate, const uint16_t* W_up,
                              const uint16_t* W_down, uint16_t* delta_emb,
                              void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* The three stages dg_self_cond_logits runs, exposed so a caller can place events or work
 * between them.  They must be called in this order, on one stream, with one workspace
 * (sized by dg_self_cond_workspace_bytes) and the same n_canvas, L, d and h:
 *   dg_self_cond_prepare: selects the canvases whose feedback is computed this step
 *                         (the list lives in the workspace) and zeroes the delta_emb rows
 *                         of all others;
 *   dg_self_cond_pe:      pe = softmax(logits / T) . E for the selected canvases, into the
 *                         workspace (the tensor-core contraction over the vocabulary);
 *   dg_self_cond_mlp:     delta_emb rows of the selected canvases from pe.
 * Arguments, limits and errors are those of dg_self_cond_logits. */
DG_API dg_status dg_self_cond_prepare(const dg_canvas_params* params, const uint8_t* converged,
                                      int64_t n_canvas, int32_t L, int32_t d, int32_t h,
                                      uint16_t* delta_emb, void* workspace, size_t workspace_bytes,
                                      dg_stream_t stream);
DG_API dg_status dg_self_cond_pe(const void* logits, dg_dtype dtype, int64_t ld, const float* lse,
                                 const dg_canvas_params* params, int64_t n_canvas, int32_t L,
                                 int64_t V, int32_t d, int32_t h, const uint16_t* E,
                                 void* workspace, size_t workspace_bytes, dg_stream_t stream);
DG_API dg_status dg_self_cond_mlp(int64_t n_canvas, int32_t L, int32_t d, int32_t h,
                                  const uint16_t* W_gate, const uint16_t* W_up,
                                  const uint16_t* W_down, uint16_t* delta_emb, void* workspace,
                                  size_t workspace_bytes, dg_stream_t stream);

/* For a feedback started before the step's convergence was known (dg_self_cond_prepare with
 * converged = NULL, while dg_denoise_accept runs on another stream): zeroes the delta_emb
 * rows of every canvas that got feedback (DG_ACTIVE and DG_SELF_COND, not DG_READ_ONLY) and
 * has converged[c] = 1, which makes delta_emb exactly what dg_self_cond_logits with that
 * converged array writes.  Call it on the feedback's stream after dg_self_cond_mlp, once the
 * converged array is complete (an event from the acceptance's stream).
 *   params (device) [n_canvas]; converged (device) [n_canvas] uint8;
 *   delta_emb (device, in/out) bf16 [n_canvas][L][d], 16-byte aligned.
 * Limits: L <= 1024, d a multiple of 8 in [8, 65536], n_canvas <= 65535 (0 launches nothing).
 * Errors: DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT, DG_ERR_CUDA. */
DG_API dg_status dg_self_cond_zero_converged(const dg_canvas_params* params, const uint8_t* converged,
                                             int64_t n_canvas, int32_t L, int32_t d,
                                             uint16_t* delta_emb, dg_stream_t stream);

/* Workspace for dg_self_cond_probs. */
DG_API size_t dg_self_cond_probs_workspace_bytes(int64_t n_rows, int32_t d, int32_t h);

/* The same feedback from caller-given probability rows (each row sums to 1):
 *   P (device) bf16 [n_rows][ld], ld >= V, ld * 2 a multiple of 16; delta_emb (device, out)
 *   bf16 [n_rows][d].  E and W as above. */
DG_API dg_status dg_self_cond_probs(const uint16_t* P, int64_t ld, int64_t n_rows, int64_t V,
                             int32_t d, int32_t h, const uint16_t* E, const uint16_t* W_gate,
                             const uint16_t* W_up, const uint16_t* W_down, uint16_t* delta_emb,
                             void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* The tensor-core GEMM engine behind the self-conditioning on plain operands:
 *   C[m][n] = sum_k A[m][k] * B(k, n), fp32 out, with B(k, n) = B[n][k] when b_mn_major = 0
 *   (B stored [N][K]) and B[k][n] when b_mn_major = 1 (B stored [K][N]).
 *   A (device) bf16 [M][lda]; B (device) bf16; C (device, out) float [M][ldc].
 *   lda, ldb multiples of 8; all pointers 16-byte aligned.  Workspace from
 *   dg_gemm_workspace_bytes(M, N). */
DG_API size_t dg_gemm_workspace_bytes(int64_t M, int64_t N);
DG_API dg_status dg_gemm_bf16(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                       int b_mn_major, float* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                       void* workspace, size_t workspace_bytes, dg_stream_t stream);

/* dg_gemm_bf16 for callers that cannot allocate device memory (no counterpart in the
 * method's description; this is a deployment aid).  Some callers may not call cudaMalloc at
 * all: a plugin whose host program hands it only input and output buffers, or code on a
 * path where an allocation (and the device synchronisation it can cause) is not allowed.
 * This variant takes no workspace: its split-K partial tiles live in a fixed array of
 * DG_NOALLOC_SCRATCH_BYTES (8 MiB) in the library's device memory, which every GPU that
 * loads the library keeps until the process exits.  The call itself allocates nothing.
 *   - Arguments, layouts, tiling and results are those of dg_gemm_bf16 (the same k-slices,
 *     so the same sums); only the workspace is gone.
 *   - Problems whose partial tiles need more than DG_NOALLOC_SCRATCH_BYTES are rejected with
 *     DG_ERR_UNSUPPORTED before anything is launched (use dg_gemm_bf16 for those).
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream capture.
 *   - Nothing in the array needs to start at zero: each partial tile is written in full
 *     before it is read.  All calls share the one array and it keeps the last call's
 *     contents, so calls that overlap on the GPU (other streams, other host threads) race:
 *     serialise them. */
#define DG_NOALLOC_SCRATCH_BYTES (8u << 20)
DG_API dg_status dg_gemm_bf16_noalloc(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                                      int b_mn_major, float* C, int64_t ldc, int64_t M, int64_t N,
                                      int64_t K, dg_stream_t stream);

/* ------------------------------------------------------------------------------------ */
/* Around the step: single-pass reads, the next pass's inputs, commit.                  */
/* ------------------------------------------------------------------------------------ */

/* Single-pass reads [SPR, "답의 내용은 몰라도 답을 담을 자리는 안다"]: a read-only request
 * reads the probability of fixed answer tokens at its answer slots.  For every position of
 * every DG_ACTIVE canvas and every slot k < C:
 *   probs[c][i][k] = exp(logits[c][i][tok] / T - lse[c][i]),  tok = choices[c][i][k],
 * the probability under the step's distribution softmax(logits / T) (T of the canvas; 1
 * for plain probabilities), with lse from dg_denoise_step of the same logits.  A slot with a
 * token outside [0, V) gives 0 (use -1 for unused slots).  Inactive canvases are skipped.
 *   logits  (device) [n_canvas][L][ld] bf16 or fp32, as for dg_denoise_step.
 *   lse     (device) [n_canvas][L] float.
 *   choices (device) [n_canvas][L][C] int32.
 *   probs   (device, out) [n_canvas][L][C] float.
 * Limits: 1 <= C <= 1024, L and V as dg_denoise_step.
 * Errors: DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT (logits not 16-byte aligned), DG_ERR_CUDA. */
DG_API dg_status dg_choice_probs(const void* logits, dg_dtype dtype, int64_t ld, const float* lse,
                          const dg_canvas_params* params, int64_t n_canvas, int32_t L, int64_t V,
                          const int32_t* choices, int32_t C, float* probs, dg_stream_t stream);

/* The next pass's canvas embeddings [DG "DiffusionGemmaModelState와 DiffusionSampler", the
 * input-preparation hook; "자기 조건화": the feedback is added to the canvas embeddings]:
 *   out[r] = bf16( fma(scale, E[canvas[r]], delta_emb[r]) )   for r < n_rows,
 * one fp32 fused multiply-add per element, rounded to nearest even.  delta_emb NULL (the
 * prefill and commit passes, no feedback) adds nothing; `scale` is the model's embedding
 * scale (1 for a plain lookup).  A token outside [0, V) gives a zero row.
 *   canvas    (device) [n_rows] int32 (e.g. the [n][L] canvas, n_rows = n * L).
 *   E         (device) [V][d] bf16.
 *   delta_emb (device, may be NULL) [n_rows][d] bf16.
 *   out       (device, out) [n_rows][d] bf16; must not overlap E or delta_emb.
 * Limits: d % 8 == 0, 8 <= d <= 65536, 0 <= n_rows < 2^31, 2 <= V < 2^31.
 * Errors: DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT (E, delta_emb, out not 16-byte aligned),
 * DG_ERR_CUDA. */
DG_API dg_status dg_embed_canvas(const int32_t* canvas, int64_t n_rows, int64_t V, const uint16_t* E,
                          int32_t d, const uint16_t* delta_emb, float scale, uint16_t* out,
                          dg_stream_t stream);

/* Commit case [DG "DiffusionGemmaModelState와 DiffusionSampler"]: every canvas that is
 * DG_ACTIVE and converged this step emits its argmax canvas as the block's tokens, and its
 * loop state is reset for the next block (prev_argmax = -1, stable_count = 0);
 * committed[c] = 1 for those canvases and 0 for every other (whose tokens and state are
 * left unchanged).  Call it after dg_denoise_step and before dg_advance_params.
 *   converged (device) [n_canvas] uint8, argmax (device) [n_canvas][L] int32.
 *   tokens, prev_argmax (device, in/out) [n_canvas][L] int32; stable_count (device, in/out)
 *   [n_canvas] int32; committed (device, out) [n_canvas] uint8.
 * Limits: 1 <= L <= 1024, 0 <= n_canvas <= 65535.  Errors: DG_ERR_INVALID_ARG, DG_ERR_CUDA. */
DG_API dg_status dg_commit(const dg_canvas_params* params, const uint8_t* converged, const int32_t* argmax,
                    int64_t n_canvas, int32_t L, int32_t* tokens, int32_t* prev_argmax,
                    int32_t* stable_count, uint8_t* committed, dg_stream_t stream);

/* ------------------------------------------------------------------------------------ */
/* Random numbers and status.                                                          */
/* ------------------------------------------------------------------------------------ */

/* Philox-4x32-10 words [PHX] for counters (block0 + b, position, step, stream | seed bits),
 * b = 0..n_blocks-1, key (lo32(seed), request_id): out (device) uint32 [n_blocks][4]. */
DG_API dg_status dg_philox_words(uint64_t seed, uint32_t request_id, uint32_t step, uint32_t position,
                          uint32_t stream_id, uint32_t block0, int64_t n_blocks, uint32_t* out,
                          dg_stream_t stream);

/* Synchronises `stream`, then returns the device status word of the current device in
 * *status (DG_DEV_* bits accumulated since the last clear). */
DG_API dg_status dg_get_device_status(dg_stream_t stream, uint32_t* status);

/* Synchronises `stream` and clears the status word of the current device. */
DG_API dg_status dg_clear_device_status(dg_stream_t stream);

/* Diagnostic hook (the method's pages have no counterpart; this checks the library's own
 * failure handling).  Runs the bounded mbarrier waits that every kernel of the library uses
 * (one thread polling, and a whole warp with one lane polling) on a shared-memory barrier
 * that never receives an arrival, with a limit of `polls` polls (1..65536, each at most
 * about a microsecond) instead of the kernels' 2^22, in one warp of one CTA on `stream`.
 * The expired waits return and raise DG_DEV_TIMEOUT in the status word, exactly as an
 * expired wait inside a kernel does; no copy or MMA is in flight, so nothing else unwinds.
 *   result (device, out) uint32 [3], 4-byte aligned: [0] the single-thread wait (0 =
 *   expired), [1] the whole-warp wait (0 = expired), [2] a wait on a barrier that did
 *   receive its arrival (1 = completed).
 * Returns DG_ERR_INVALID_ARG for polls outside 1..65536 or a null result (nothing
 * launched). */
DG_API dg_status dg_probe_bounded_wait(uint32_t polls, uint32_t* result, dg_stream_t stream);

/* Static, human-readable name of a status code. */
DG_API const char* dg_status_string(dg_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
DG_API int32_t dg_version(void);

/* Number of kernel launches the library has enqueued in this process so far (all devices). */
DG_API uint64_t dg_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
