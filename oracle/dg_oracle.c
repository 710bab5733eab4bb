/*
 * dg_oracle.c -- plain, slow, fp64 CPU oracle of the entropy-bounded denoising step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  It shares no code, header, table or
 * constant generator with the CUDA library; it is written from the method's
 * description, not from the kernels.
 *
 * Sources (web pages, cited by title and section):
 *   [DG]  "DiffusionGemma: vLLM이 네이티브로 지원하는 최초의 디퓨전 언어 모델(dLLM)"
 *         (discuss.pytorch.kr), sections "엔트로피 기반 디노이징" (entropy-based
 *         denoising, with the equation H(p) = -sum_i p_i log p_i), "자기 조건화"
 *         (self-conditioning) and "DiffusionGemmaModelState와 DiffusionSampler"
 *         (the Prefill / Denoise / Commit cases of the sampler step).
 *   [SPR] "답은 한 번 읽는데 모델은 왜 두 번 돌까? DiffusionGemma의 실행 경로 합치기"
 *         (single-pass reads), paragraph on request eligibility
 *         (diffusion_read_only and diffusion_max_steps = 1).
 *   [PHX] J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel random numbers: as easy
 *         as 1, 2, 3", SC'11 -- the Philox-4x32 bijection with 10 rounds.
 *   [GELU] D. Hendrycks, K. Gimpel, "Gaussian Error Linear Units" -- tanh form.
 *
 * Where the pages are silent, the reading taken is stated at the function that takes
 * it.  Everything is fp64 (except where an output is a rounded bf16 bit pattern, whose
 * definition fixes the rounding) and follows the definitions in the order the pages
 * give them; nothing is blocked, fused or reordered.
 *
 * Pins: every function here is checked by tests/test_oracle_*.py against closed
 * forms, hand-worked examples, brute force and invariants (see those files).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------- */
/* Counter-based random numbers: Philox-4x32 [PHX].                                 */
/* One round maps (X0,X1,X2,X3) with round key (K0,K1) to                           */
/*   (hi(M1*X2) ^ X1 ^ K0,  lo(M1*X2),  hi(M0*X0) ^ X3 ^ K1,  lo(M0*X0)),           */
/* and the key is advanced by the Weyl constants between rounds.                    */
/* ------------------------------------------------------------------------------- */
static const uint32_t PHX_M0 = 0xD2511F53u;
static const uint32_t PHX_M1 = 0xCD9E8D57u;
static const uint32_t PHX_W0 = 0x9E3779B9u; /* golden ratio */
static const uint32_t PHX_W1 = 0xBB67AE85u; /* sqrt(3) - 1  */

void orc_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds, uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < rounds; ++r) {
        if (r > 0) { k0 += PHX_W0; k1 += PHX_W1; }
        uint64_t p0 = (uint64_t)PHX_M0 * (uint64_t)x0;
        uint64_t p1 = (uint64_t)PHX_M1 * (uint64_t)x2;
        uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;
        uint32_t y1 = (uint32_t)p1;
        uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
        uint32_t y3 = (uint32_t)p0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Random-number contract shared (by specification, not by code) with the kernels:
 *   key     = (lo32(seed), request_id)
 *   counter = (block, position, step, stream | (bits 32..55 of seed) << 8)
 *   streams: 0 = Gumbel noise, 1 = renoise tokens, 2 = canvas initialisation.   */
enum { ORC_STREAM_GUMBEL = 0, ORC_STREAM_RENOISE = 1, ORC_STREAM_INIT = 2 };

static void orc_draw(uint64_t seed, uint32_t request_id, uint32_t block, uint32_t position,
                     uint32_t step, uint32_t stream, uint32_t out[4])
{
    uint32_t ctr[4] = { block, position, step,
                        stream | ((uint32_t)((seed >> 32) & 0xFFFFFFu) << 8) };
    uint32_t key[2] = { (uint32_t)(seed & 0xFFFFFFFFu), request_id };
    orc_philox4x32(ctr, key, 10, out);
}

/* Uniform in (0,1): the top 23 bits of a word, centred in their cell:
 * u = (floor(w / 2^9) + 1/2) / 2^23, so 2^-24 <= u <= 1 - 2^-24 and u is exact in fp32. */
double orc_uniform(uint32_t w)
{
    return ((double)(w >> 9) + 0.5) * (1.0 / 8388608.0);
}

/* Uniform token in [0, V): floor(x * V / 2^64) with x the 64-bit word (w0 << 32 | w1). */
uint32_t orc_token(uint32_t w0, uint32_t w1, uint32_t V)
{
    unsigned __int128 x = ((unsigned __int128)w0 << 32) | (unsigned __int128)w1;
    return (uint32_t)((x * (unsigned __int128)V) >> 64);
}

/* Gumbel noise g = -log(-log u) for vocabulary entry v of one canvas position. */
double orc_gumbel(uint64_t seed, uint32_t request_id, uint32_t step, uint32_t position, uint32_t v)
{
    uint32_t w[4];
    orc_draw(seed, request_id, v >> 2, position, step, ORC_STREAM_GUMBEL, w);
    double u = orc_uniform(w[v & 3u]);
    return -log(-log(u));
}

/* Uniform token for renoising (stream 1) or for a fresh canvas (stream 2). */
uint32_t orc_random_token(uint64_t seed, uint32_t request_id, uint32_t step, uint32_t position,
                          uint32_t stream, uint32_t V)
{
    uint32_t w[4];
    orc_draw(seed, request_id, 0u, position, step, stream, w);
    return orc_token(w[0], w[1], V);
}

/* ------------------------------------------------------------------------------- */
/* Logit access.  dtype 0 = bf16 (raw 16-bit patterns), 1 = fp32.                   */
/* ------------------------------------------------------------------------------- */
static double orc_logit(const void* row, int dtype, int64_t v)
{
    if (dtype == 0) {
        uint32_t bits = (uint32_t)((const uint16_t*)row)[v] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)row)[v];
}

/* ------------------------------------------------------------------------------- */
/* Per-position statistics [DG, "엔트로피 기반 디노이징" and the Denoise case].      */
/* ------------------------------------------------------------------------------- */
typedef struct {
    double entropy;     /* H(p) = -sum_{p_v > 0} p_v log p_v, p = softmax(x / T)           */
    double entropy_alt; /* the same quantity as log(c + r) + (-t) / (c + r), see below     */
    double lse;         /* log sum_v exp(x_v / T)                                          */
    double score1;      /* largest perturbed score x_v / T + g_v                           */
    double score2;      /* second largest perturbed score                                  */
    int32_t argmax;     /* smallest v with x_v = max x (raw logits; T > 0 keeps the order) */
    int32_t sample;     /* smallest v attaining score1; -1 when not sampled                */
    int32_t nonfinite;  /* number of NaN or +inf logits in the row                         */
    int32_t pad;
} orc_row_result;

/* One canvas position.  Steps, as the Denoise case states them:
 *   1. scale the logits by the temperature: y_v = x_v / T;
 *   2. p = softmax(y); H(p) = -sum p log p (the entropy equation);
 *   3. the best-guess token is argmax x (it is what a converged canvas commits);
 *   4. the candidate token is the Gumbel-max sample argmax_v (y_v + g_v).
 * Reading: the same temperature-scaled distribution gives H, the sample and (in the
 * self-conditioning step) P; the argmax is taken on the raw logits, which T > 0 does
 * not reorder.  Exact ties go to the lowest index. */
void orc_row_stats(const void* row, int dtype, int64_t V, double T, uint64_t seed,
                   uint32_t request_id, uint32_t step, uint32_t position, int do_sample,
                   orc_row_result* res)
{
    memset(res, 0, sizeof *res);
    res->sample = -1;
    res->score1 = -INFINITY;
    res->score2 = -INFINITY;

    /* max of the raw logits and the lowest index attaining it */
    double xmax = -INFINITY;
    int64_t amax = 0;
    int32_t nonfinite = 0;
    for (int64_t v = 0; v < V; ++v) {
        double x = orc_logit(row, dtype, v);
        if (isnan(x) || x == INFINITY) { ++nonfinite; continue; }
        if (x > xmax) { xmax = x; amax = v; }
    }
    res->argmax = (int32_t)amax;
    res->nonfinite = nonfinite;

    /* softmax of y = x / T, written with the max subtracted */
    double m = xmax / T;
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double y = orc_logit(row, dtype, v) / T;
        s += exp(y - m);
    }
    res->lse = m + log(s);

    /* H(p) = -sum_{p > 0} p log p */
    double H = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double y = orc_logit(row, dtype, v) / T;
        double p = exp(y - m) / s;
        if (p > 0.0) H -= p * log(p);
    }
    res->entropy = H;

    /* The same entropy through the split used to keep near-one-hot rows accurate:
     * with z_v = y_v - m, c = #{z_v = 0}, r = sum_{z_v < 0} e^{z_v}, t = sum e^{z_v} z_v,
     * H = log(c + r) - t / (c + r).  (Substitute p_v = e^{z_v} / (c + r) into H.) */
    double c = 0.0, r = 0.0, t = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double z = orc_logit(row, dtype, v) / T - m;
        if (z == 0.0) c += 1.0;
        else if (z < 0.0) { double e = exp(z); if (e > 0.0) { r += e; t += e * z; } }
    }
    res->entropy_alt = (c == 1.0 ? log1p(r) : log(c + r)) - t / (c + r);

    if (!do_sample) return;

    /* Gumbel-max: sample = argmax_v (y_v + g_v), g_v = -log(-log u_v). */
    double b1 = -INFINITY, b2 = -INFINITY;
    int64_t i1 = -1;
    for (int64_t v = 0; v < V; ++v) {
        double x = orc_logit(row, dtype, v);
        if (isnan(x)) continue;
        double score = x / T + orc_gumbel(seed, request_id, step, position, (uint32_t)v);
        if (score > b1) { b2 = b1; b1 = score; i1 = v; }
        else if (score > b2) { b2 = score; }
    }
    res->sample = (int32_t)i1;
    res->score1 = b1;
    res->score2 = b2;
}

/* ------------------------------------------------------------------------------- */
/* Entropy-bound acceptance [DG, "엔트로피 기반 디노이징"]: walk the positions from   */
/* most to least confident (ascending H, ties by position) and accept tokens until  */
/* just before the cumulative entropy would exceed the budget beta.                 */
/* Readings: "just before exceeding" = accept while the running sum stays <= beta;  */
/* at least min_accept positions are accepted (0 or 1).                             */
/* ------------------------------------------------------------------------------- */
typedef struct { double h; int32_t idx; } orc_key;

static int orc_key_cmp(const void* a, const void* b)
{
    const orc_key* x = (const orc_key*)a;
    const orc_key* y = (const orc_key*)b;
    if (x->h < y->h) return -1;
    if (x->h > y->h) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

/* Returns the number accepted.  order (optional, [L]) receives the sorted positions;
 * cut_gap (optional) receives the relative entropy gap between the last accepted and
 * the first rejected position; budget_gap (optional) the smaller of
 * |S_last_accepted - beta| / beta and |S_first_rejected - beta| / beta over the prefix
 * sums S that decided the cut (+inf where a side does not exist). */
int32_t orc_accept(const double* H, int32_t L, double beta, int32_t min_accept,
                   uint8_t* accept_mask, int32_t* order, double* cut_gap, double* budget_gap)
{
    orc_key* keys = (orc_key*)malloc(sizeof(orc_key) * (size_t)(L > 0 ? L : 1));
    for (int32_t i = 0; i < L; ++i) { keys[i].h = H[i]; keys[i].idx = i; }
    qsort(keys, (size_t)L, sizeof(orc_key), orc_key_cmp);

    int32_t n_budget = 0;
    double S = 0.0, S_last = NAN, S_next = NAN;
    for (int32_t j = 0; j < L; ++j) {
        double S_new = S + keys[j].h;
        if (S_new <= beta) { S = S_new; S_last = S; ++n_budget; }
        else { S_next = S_new; break; }
    }
    int32_t n_acc = n_budget;
    if (n_acc < min_accept) n_acc = min_accept;
    if (n_acc > L) n_acc = L;

    for (int32_t i = 0; i < L; ++i) accept_mask[i] = 0;
    for (int32_t j = 0; j < n_acc; ++j) accept_mask[keys[j].idx] = 1;
    if (order) for (int32_t j = 0; j < L; ++j) order[j] = keys[j].idx;

    if (cut_gap) {
        double g = INFINITY;
        if (n_acc > 0 && n_acc < L) {
            double a = keys[n_acc - 1].h, b = keys[n_acc].h;
            double den = fmax(fabs(a), fabs(b));
            g = den > 0.0 ? fabs(b - a) / den : 0.0;
        }
        *cut_gap = g;
    }
    if (budget_gap) {
        double g = INFINITY;
        double den = fabs(beta) > 0.0 ? fabs(beta) : 1.0;
        if (!isnan(S_last)) g = fmin(g, fabs(S_last - beta) / den);
        if (!isnan(S_next)) g = fmin(g, fabs(S_next - beta) / den);
        *budget_gap = g;
    }
    free(keys);
    return n_acc;
}

/* ------------------------------------------------------------------------------- */
/* One denoise step over n canvases [DG, Denoise case and convergence paragraph].   */
/* Per-canvas parameters are given as separate arrays.  flags: 1 ACTIVE,            */
/* 2 READ_ONLY, 4 SELF_COND.  Layouts: logits [n][L][ld], everything else [n][L]    */
/* or [n].  Inactive canvases are neither read nor written.                         */
/* Readings: every position is resampled each step; accepted positions take this    */
/* step's sample; rejected ones take a uniform token over [0, V) (renoise stream);  */
/* the convergence history is the previous argmax canvas plus a count of            */
/* consecutive unchanged steps; the step cap converges when step + 1 >= S.  A       */
/* read-only canvas ([SPR]: read-only with a single step) only reads its statistics:*/
/* nothing is accepted, the canvas is left as it is and it is converged.            */
/* ------------------------------------------------------------------------------- */
enum { ORC_ACTIVE = 1u, ORC_READ_ONLY = 2u, ORC_SELF_COND = 4u };

void orc_denoise_step(const void* logits, int dtype, int64_t ld, int64_t n, int32_t L, int64_t V,
                      const float* temperature, const float* beta, const float* tau,
                      const int32_t* k, const int32_t* max_steps, const int32_t* min_accept,
                      const int32_t* step, const uint32_t* request_id, const uint32_t* flags,
                      uint64_t seed,
                      int32_t* canvas, int32_t* prev_argmax, int32_t* stable_count,
                      uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                      double* entropy, double* lse, uint8_t* converged,
                      double* mean_entropy, int32_t* n_accept,
                      double* sample_gap, double* cut_gap, double* budget_gap, double* tau_gap,
                      int n_threads)
{
    size_t esize = dtype == 0 ? 2 : 4;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    /* the per-position statistics are independent: one row at a time, in parallel */
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < n * (int64_t)L; ++q) {
        int64_t c = q / L;
        int32_t i = (int32_t)(q % L);
        if (!(flags[c] & ORC_ACTIVE)) continue;
        int read_only = (flags[c] & ORC_READ_ONLY) != 0;
        const char* row = (const char*)logits + (size_t)q * (size_t)ld * esize;
        orc_row_result res;
        orc_row_stats(row, dtype, V, (double)temperature[c], seed, request_id[c],
                      (uint32_t)step[c], (uint32_t)i, !read_only, &res);
        entropy[q] = res.entropy;
        lse[q] = res.lse;
        argmax[q] = res.argmax;
        sample[q] = res.sample;
        if (sample_gap) {
            double den = fabs(res.score1) > 1.0 ? fabs(res.score1) : 1.0;
            sample_gap[q] = read_only ? INFINITY : (res.score1 - res.score2) / den;
        }
    }

    for (int64_t c = 0; c < n; ++c) {
        if (!(flags[c] & ORC_ACTIVE)) continue;
        int read_only = (flags[c] & ORC_READ_ONLY) != 0;
        int64_t base = c * (int64_t)L;

        /* acceptance and renoise */
        int32_t nacc = 0;
        double cg = INFINITY, bg = INFINITY;
        if (read_only) {
            for (int32_t i = 0; i < L; ++i) accept_mask[base + i] = 0;
        } else {
            nacc = orc_accept(entropy + base, L, (double)beta[c], min_accept[c],
                              accept_mask + base, NULL, &cg, &bg);
            for (int32_t i = 0; i < L; ++i) {
                if (accept_mask[base + i]) canvas[base + i] = sample[base + i];
                else canvas[base + i] = (int32_t)orc_random_token(seed, request_id[c],
                        (uint32_t)step[c], (uint32_t)i, ORC_STREAM_RENOISE, (uint32_t)V);
            }
        }
        if (n_accept) n_accept[c] = nacc;
        if (cut_gap) cut_gap[c] = cg;
        if (budget_gap) budget_gap[c] = bg;

        /* convergence: argmax unchanged for k consecutive steps AND mean entropy < tau,
         * or the step cap */
        int same = 1;
        for (int32_t i = 0; i < L; ++i)
            if (argmax[base + i] != prev_argmax[base + i]) { same = 0; break; }
        int32_t st = same ? stable_count[c] + 1 : 0;
        double Hsum = 0.0;
        for (int32_t i = 0; i < L; ++i) Hsum += entropy[base + i];
        double Hbar = Hsum / (double)L;
        int conv = (st >= k[c] && Hbar < (double)tau[c]) || (step[c] + 1 >= max_steps[c]);
        if (read_only) conv = 1;
        converged[c] = (uint8_t)conv;
        stable_count[c] = st;
        for (int32_t i = 0; i < L; ++i) prev_argmax[base + i] = argmax[base + i];
        if (mean_entropy) mean_entropy[c] = Hbar;
        if (tau_gap) tau_gap[c] = fabs(Hbar - (double)tau[c]) / fmax(fabs((double)tau[c]), 1e-300);
    }
}

/* Prefill case [DG, "DiffusionGemmaModelState와 DiffusionSampler"]: a fresh canvas of
 * uniform random tokens (stream 2) for every active canvas. */
void orc_canvas_init(int32_t* canvas, int64_t n, int32_t L, int64_t V, const int32_t* step,
                     const uint32_t* request_id, const uint32_t* flags, uint64_t seed)
{
    for (int64_t c = 0; c < n; ++c) {
        if (!(flags[c] & ORC_ACTIVE)) continue;
        for (int32_t i = 0; i < L; ++i)
            canvas[c * L + i] = (int32_t)orc_random_token(seed, request_id[c], (uint32_t)step[c],
                                                          (uint32_t)i, ORC_STREAM_INIT, (uint32_t)V);
    }
}

/* ------------------------------------------------------------------------------- */
/* Self-conditioning [DG, "자기 조건화"]: the previous step's full softmax P is       */
/* turned into a probability-weighted mean of the token embeddings, pe = P . E,     */
/* then passed through a small gated MLP whose output is added to the next pass's   */
/* canvas embeddings.                                                               */
/* Reading: delta = W_down (act(W_gate pe) * (W_up pe)), no bias, no norm,          */
/* act = GELU, tanh form [GELU]; W_gate, W_up are [h][d], W_down is [d][h] (row =   */
/* output unit).  E and W are bf16 bit patterns, widened exactly to fp64.           */
/* ------------------------------------------------------------------------------- */
static double orc_bf16(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

double orc_gelu_tanh(double z)
{
    const double k = sqrt(2.0 / M_PI);
    return 0.5 * z * (1.0 + tanh(k * (z + 0.044715 * z * z * z)));
}

/* pe[r][j] = sum_v P[r][v] E[v][j] for given probability rows (fp64 in). */
void orc_pe_from_probs(const double* P, int64_t n_rows, int64_t V, int32_t d,
                       const uint16_t* E, double* pe, int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        double* out = pe + r * d;
        for (int32_t j = 0; j < d; ++j) out[j] = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            double p = P[r * V + v];
            if (p == 0.0) continue;
            const uint16_t* e = E + v * d;
            for (int32_t j = 0; j < d; ++j) out[j] += p * orc_bf16(e[j]);
        }
    }
}

/* delta[r] = W_down (gelu(W_gate pe[r]) * (W_up pe[r])) */
void orc_gated_mlp(const double* pe, int64_t n_rows, int32_t d, int32_t h,
                   const uint16_t* W_gate, const uint16_t* W_up, const uint16_t* W_down,
                   double* delta, int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const double* z = pe + r * d;
        double* hid = (double*)malloc(sizeof(double) * (size_t)h);
        for (int32_t a = 0; a < h; ++a) {
            double g = 0.0, u = 0.0;
            for (int32_t j = 0; j < d; ++j) {
                g += orc_bf16(W_gate[(int64_t)a * d + j]) * z[j];
                u += orc_bf16(W_up[(int64_t)a * d + j]) * z[j];
            }
            hid[a] = orc_gelu_tanh(g) * u;
        }
        for (int32_t j = 0; j < d; ++j) {
            double o = 0.0;
            for (int32_t a = 0; a < h; ++a) o += orc_bf16(W_down[(int64_t)j * h + a]) * hid[a];
            delta[r * d + j] = o;
        }
        free(hid);
    }
}

/* Softmax rows from logits: P[r][v] = exp(x_v / T - lse), with lse computed here
 * from the definition (the oracle never takes a statistic from elsewhere). */
void orc_probs_from_logits(const void* logits, int dtype, int64_t ld, int64_t n_rows,
                           int64_t V, const double* T_rows, double* P, int n_threads)
{
    size_t esize = dtype == 0 ? 2 : 4;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const char* row = (const char*)logits + (size_t)r * (size_t)ld * esize;
        double T = T_rows[r];
        double m = -INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            double y = orc_logit(row, dtype, v) / T;
            if (y > m) m = y;
        }
        double s = 0.0;
        for (int64_t v = 0; v < V; ++v) s += exp(orc_logit(row, dtype, v) / T - m);
        double lse = m + log(s);
        for (int64_t v = 0; v < V; ++v) P[r * V + v] = exp(orc_logit(row, dtype, v) / T - lse);
    }
}

/* ------------------------------------------------------------------------------- */
/* Single-pass reads [SPR], sections "답의 내용은 몰라도 답을 담을 자리는 안다" and     */
/* "12개 입력과 4개 캔버스를 예산에 넣어 보면": a read-only request wants the        */
/* probability of fixed answer tokens at its answer slots.  Reading: the probability */
/* under the step's distribution softmax(x / T), p = exp(x_tok / T - lse), with lse   */
/* from the definition; slots with a token outside [0, V) (unused: -1) give 0.        */
/* ------------------------------------------------------------------------------- */
void orc_choice_probs(const void* logits, int dtype, int64_t ld, int64_t n_rows, int64_t V,
                      const double* T_rows, const int32_t* choices, int32_t C, double* probs,
                      int n_threads)
{
    size_t esize = dtype == 0 ? 2 : 4;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const char* row = (const char*)logits + (size_t)r * (size_t)ld * esize;
        double T = T_rows[r];
        double m = -INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            double y = orc_logit(row, dtype, v) / T;
            if (y > m) m = y;
        }
        double s = 0.0;
        for (int64_t v = 0; v < V; ++v) s += exp(orc_logit(row, dtype, v) / T - m);
        double lse = m + log(s);
        for (int32_t k = 0; k < C; ++k) {
            int32_t tok = choices[r * C + k];
            probs[r * C + k] = (tok >= 0 && tok < V) ? exp(orc_logit(row, dtype, tok) / T - lse) : 0.0;
        }
    }
}

/* ------------------------------------------------------------------------------- */
/* Step-after glue [DG], section "DiffusionGemmaModelState와 DiffusionSampler" (the   */
/* input-preparation hook adds the stored feedback to the canvas embeddings) and     */
/* "자기 조건화" (the feedback is added to the next pass's canvas embeddings):       */
/*   emb[r] = bf16( fma(scale, E[canvas[r]], delta[r]) )                            */
/* The output is a bf16 bit pattern, so its definition fixes the rounding: one fp32  */
/* fused multiply-add, then round-to-nearest-even to bf16.  `scale` is the model's    */
/* embedding scale (1 for a plain lookup); delta NULL (prefill / commit passes: no   */
/* feedback) adds nothing.  A token outside [0, V) gives a zero row.                 */
/* ------------------------------------------------------------------------------- */
uint16_t orc_bf16_round(float f)
{
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    if ((b & 0x7f800000u) == 0x7f800000u && (b & 0x007fffffu) != 0u)
        return (uint16_t)((b >> 16) | 0x0040u);          /* NaN stays NaN (quiet) */
    uint32_t lsb = (b >> 16) & 1u;                       /* ties go to the even neighbour */
    return (uint16_t)((b + 0x7fffu + lsb) >> 16);
}

void orc_embed_canvas(const int32_t* canvas, int64_t n_rows, int64_t V, const uint16_t* E,
                      int32_t d, const uint16_t* delta, float scale, uint16_t* out)
{
    for (int64_t r = 0; r < n_rows; ++r) {
        int32_t tok = canvas[r];
        for (int32_t j = 0; j < d; ++j) {
            if (tok < 0 || tok >= V) {
                out[r * d + j] = 0;
                continue;
            }
            float e = (float)orc_bf16(E[(int64_t)tok * d + j]);
            float a = delta ? (float)orc_bf16(delta[r * d + j]) : 0.0f;
            out[r * d + j] = orc_bf16_round(fmaf(scale, e, a));
        }
    }
}

/* ------------------------------------------------------------------------------- */
/* Commit [DG], section "DiffusionGemmaModelState와 DiffusionSampler", Commit case:  */
/* a converged canvas emits its argmax as the block's tokens.  Reading: only         */
/* canvases still active this step commit (a canvas commits once); their loop state  */
/* is reset for the next block (no previous argmax, stable count 0).                  */
/* ------------------------------------------------------------------------------- */
void orc_commit(const uint8_t* converged, const uint8_t* active, const int32_t* argmax, int64_t n,
                int32_t L, int32_t* tokens, int32_t* prev_argmax, int32_t* stable_count,
                uint8_t* committed)
{
    for (int64_t c = 0; c < n; ++c) {
        int go = active[c] && converged[c];
        committed[c] = (uint8_t)(go ? 1 : 0);
        if (!go) continue;
        for (int32_t i = 0; i < L; ++i) {
            tokens[c * L + i] = argmax[c * L + i];
            prev_argmax[c * L + i] = -1;
        }
        stable_count[c] = 0;
    }
}

/* ------------------------------------------------------------------------------- */
/* LM head: the logits the denoise step reads are the model's output over the canvas */
/* [DG], section "엔트로피 기반 디노이징" (each step runs the model on the canvas and   */
/* reads the per-position distributions).  Reading (the pages do not describe the    */
/* output layer): a plain linear map of the last hidden states,                      */
/*   logits[r][v] = sum_j hidden[r][j] W[v][j],   W = [V][d] (row = vocabulary entry; */
/* the input embedding table when the model ties the two, as the Gemma family does), */
/* with no bias and no soft-capping.  The logits are stored as bf16, so their        */
/* definition fixes the rounding: the dot product, rounded once to the nearest bf16, */
/* ties to even.  The dot product is summed in fp64 (exact for small-integer          */
/* operands; otherwise within d 2^-53 sum_j |hidden[r][j] W[v][j]|).                  */
/* ------------------------------------------------------------------------------- */
/* The bf16 bit pattern nearest to x (ties to even), from x itself: no intermediate   */
/* fp32 rounding.  bf16 keeps 8 significant bits down to 2^-126 and a fixed quantum   */
/* of 2^-133 below; magnitudes that round past (2 - 2^-7) 2^127 become infinite.      */
uint16_t orc_bf16_round_f64(double x)
{
    if (isnan(x)) return (uint16_t)0x7fc0u;
    uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0u;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7f80u);
    int e;
    (void)frexp(a, &e);            /* a = m 2^e with m in [0.5, 1) */
    int q = e - 8;                 /* exponent of the quantum at a's binade */
    if (q < -133) q = -133;
    /* nearbyint rounds to nearest, ties to even (the default rounding mode) */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r > 0x1.fep127) return (uint16_t)(sign | 0x7f80u);
    float f = (float)r;            /* exact: r has at most 8 significant bits */
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    return (uint16_t)(sign | (uint16_t)(b >> 16));
}

/* logits (bf16 bits) [n_rows][ld] from hidden [n_rows][ldh] and W [V][ldw], both bf16 */
/* bits; optionally the unrounded dot products `exact` and sum_j |h_j W_vj| `abssum`  */
/* ([n_rows][V] each, may be NULL).                                                   */
void orc_lm_head_logits(const uint16_t* hidden, int64_t n_rows, int32_t d, int64_t ldh,
                        const uint16_t* W, int64_t V, int64_t ldw, uint16_t* logits, int64_t ld,
                        double* exact, double* abssum, int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    #pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int64_t v = 0; v < V; ++v) {
            double s = 0.0, sa = 0.0;
            for (int32_t j = 0; j < d; ++j) {
                double t = orc_bf16(hidden[r * ldh + j]) * orc_bf16(W[v * ldw + j]);
                s += t;
                sa += fabs(t);
            }
            logits[r * ld + v] = orc_bf16_round_f64(s);
            if (exact) exact[r * V + v] = s;
            if (abssum) abssum[r * V + v] = sa;
        }
    }
}

/* ------------------------------------------------------------------------------- */
/* Attention with per-sequence causality and a symmetric window [DG], sections        */
/* "시퀀스별로 동적으로 바뀌는 인과 어텐션" (per-sequence dynamic causal attention) and  */
/* "슬라이딩 윈도우 어텐션도 대칭으로" (the sliding window made symmetric).  A batch     */
/* mixes requests: a causal one (prefill or commit pass) lets query i see keys j <= its */
/* own position; a bidirectional one (a denoising canvas) lets every query see every   */
/* key of its sequence, context and canvas alike.  With a window W >= 0 a causal query */
/* sees keys in [pos - W, pos] and a bidirectional one keys in [pos - W, pos + W].      */
/* Reading (the pages give only the figures): a sequence's queries are its last q_len  */
/* tokens, so query i sits at position kv_len - q_len + i; scores are scale * q . k    */
/* (no soft-capping); one key/value head serves Hq / Hkv consecutive query heads.      */
/*   o[i][h] = sum_j softmax_j(scale q_i . k_j over the allowed j) v_j,               */
/*   lse[i][h] = log sum_j exp(scale q_i . k_j) over the allowed j.                   */
/* q [total_q][Hq][D], k and v [total_kv][Hkv][D] as bf16 bits; o and lse in fp64.     */
/* A query with no allowed key gets o = 0 and lse = -inf.                             */
/* ------------------------------------------------------------------------------- */
int orc_attn_allowed(int causal, int64_t window, int64_t pos, int64_t j, int64_t kv_len)
{
    if (j < 0 || j >= kv_len) return 0;
    if (causal && j > pos) return 0;
    if (window >= 0) {
        if (j < pos - window) return 0;
        if (!causal && j > pos + window) return 0;
    }
    return 1;
}

void orc_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* cu_q,
                   const int32_t* cu_kv, const uint8_t* causal, int32_t n_seq, int32_t Hq, int32_t Hkv,
                   int32_t D, int64_t window, double scale, double* o, double* lse, int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int32_t group = Hq / Hkv;
    for (int32_t s = 0; s < n_seq; ++s) {
        int64_t q0 = cu_q[s], q_len = cu_q[s + 1] - cu_q[s];
        int64_t k0 = cu_kv[s], kv_len = cu_kv[s + 1] - cu_kv[s];
        #pragma omp parallel for collapse(2) schedule(dynamic, 4)
        for (int64_t i = 0; i < q_len; ++i) {
            for (int32_t h = 0; h < Hq; ++h) {
                int64_t pos = kv_len - q_len + i;
                int32_t hk = h / group;
                const uint16_t* qi = q + ((q0 + i) * Hq + h) * D;
                double* oi = o + ((q0 + i) * Hq + h) * D;
                double* sc = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
                double m = -INFINITY;
                for (int64_t j = 0; j < kv_len; ++j) {
                    sc[j] = -INFINITY;
                    if (!orc_attn_allowed(causal[s], window, pos, j, kv_len)) continue;
                    const uint16_t* kj = k + ((k0 + j) * Hkv + hk) * D;
                    double dot = 0.0;
                    for (int32_t c = 0; c < D; ++c) dot += orc_bf16(qi[c]) * orc_bf16(kj[c]);
                    sc[j] = scale * dot;
                    if (sc[j] > m) m = sc[j];
                }
                for (int32_t c = 0; c < D; ++c) oi[c] = 0.0;
                if (m == -INFINITY) {
                    lse[(q0 + i) * Hq + h] = -INFINITY;
                    free(sc);
                    continue;
                }
                double sum = 0.0;
                for (int64_t j = 0; j < kv_len; ++j) {
                    if (sc[j] == -INFINITY) continue;
                    double w = exp(sc[j] - m);
                    sum += w;
                    const uint16_t* vj = v + ((k0 + j) * Hkv + hk) * D;
                    for (int32_t c = 0; c < D; ++c) oi[c] += w * orc_bf16(vj[c]);
                }
                for (int32_t c = 0; c < D; ++c) oi[c] /= sum;
                lse[(q0 + i) * Hq + h] = m + log(sum);
                free(sc);
            }
        }
    }
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
