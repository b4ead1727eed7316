/*
 * sampler_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of the per-decode-step token
 * sampler. Only tests/, the package's smoke() self-check and bench.py's CPU
 * baseline may load it; the product path never does. It shares no code, header,
 * table or constant generator with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *  [NOTE]  xbrilliance.ai note "采样参数对解码开销的影响：temperature、top_p 与采样核路径"
 *          (Effect of sampling parameters on decode cost), sections
 *          "解码一步里采样做什么" (what sampling does in one decode step: the fixed stage
 *          order), "哪些参数会额外打开一趟全词表计算" (which parameters open an extra
 *          full-vocab pass: defaults and the penalty / top-k / top-p / min-p stages),
 *          "采样类型与选路" (sampling type and routing: GREEDY below 1e-5, RANDOM_SEED),
 *          "best_of 与 n 的放大" (forks sample several tokens from one row).
 *  [CHECK] dev.to "SGLang's +75% sampler speedup skips Qwen3 chat requests",
 *          section "Nine lines, and exactly one call site" (Gumbel-max: argmax of
 *          probs / Exp(1) draws, same distribution as a categorical draw).
 *  [MANUAL] aiengineeringfromscratch.com "manual-sglang-101", section
 *          "Logprobs are temperature-scaled" (returned logprobs are log_softmax(l / T)).
 *
 * Arithmetic: penalties in IEEE single precision in a fixed order (compile with
 * -ffp-contract=off so no multiply-add is fused); everything after the penalties
 * (temperature, softmax, cumulative sums, the Gumbel scores) in double. Full
 * sort per row (qsort on (value desc, index asc)), explicit cumulative sums.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - penalty formulas: repetition divides positive / multiplies non-positive
 *    logits of tokens seen before, then frequency subtracts f * count, then
 *    presence subtracts p once for tokens seen before. Parity unpinned: no page
 *    prints these formulas or a worked example, so only hand-computed cases of
 *    this reading check them;
 *  - greedy when T < 1e-5 ([NOTE] sampling type); outputs of greedy rows use T = 1;
 *  - top-k keeps exactly k tokens in (value desc, index asc) order; -1 or k >= V
 *    keeps all;
 *  - top-p keeps, over the top-k set, the tokens whose exclusive prefix mass in
 *    that order is < p (always at least one);
 *  - min-p keeps tokens with p_v >= min_p * p_max, i.e. y_v - y_max >= ln(min_p);
 *  - Gumbel-max over the kept set, E_v = -ln(u_v), u_v from Philox4x32-10:
 *    key = seed (lo, hi), counter = (v >> 2, stream, offset lo, offset hi),
 *    word v & 3, u = (2 * (word >> 9) + 1) * 2^-24; ties go to the lowest index.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORACLE_DTYPE_F32 0
#define ORACLE_DTYPE_BF16 1

#define ST_OK 0
#define ST_NONFINITE 1
#define ST_ALL_NEG_INF 2
#define ST_BAD_PARAM 3
#define ST_BAD_HISTORY 4

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 and Philox4x64-10, written from the round function of        */
/* Salmon et al., SC'11 ("Parallel Random Numbers: As Easy as 1, 2, 3"):      */
/* each round multiplies counter words 0 and 2 by fixed constants, swaps the  */
/* halves into the other lanes xored with the key, and the key is bumped by   */
/* the Weyl constants between rounds.                                          */
/* ------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(prod1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)prod1;
        uint32_t n2 = (uint32_t)(prod0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)prod0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 64-bit-word member of the same family; used only to check the round
 * structure against an independent library implementation. */
void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B97F4A7C15ull;
            k1 += 0xBB67AE8584CAA73Bull;
        }
        unsigned __int128 prod0 = (unsigned __int128)0xD2E7470EE14C6C93ull * c0;
        unsigned __int128 prod1 = (unsigned __int128)0xCA5A826395121157ull * c2;
        uint64_t n0 = (uint64_t)(prod1 >> 64) ^ c1 ^ k0;
        uint64_t n1 = (uint64_t)prod1;
        uint64_t n2 = (uint64_t)(prod0 >> 64) ^ c3 ^ k1;
        uint64_t n3 = (uint64_t)prod0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32-bit Philox word that drives token v of a row. */
uint32_t oracle_noise_word(uint64_t key, uint32_t stream, uint64_t offset, int64_t v)
{
    uint32_t ctr[4] = {(uint32_t)((uint64_t)v >> 2), stream, (uint32_t)offset,
                       (uint32_t)(offset >> 32)};
    uint32_t k[2] = {(uint32_t)key, (uint32_t)(key >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, k, out);
    return out[v & 3];
}

/* Uniform in (0, 1) from the top 23 bits of a word: odd multiples of 2^-24. */
double oracle_uniform(uint32_t word)
{
    return (2.0 * (double)(word >> 9) + 1.0) * 0x1p-24;
}

/* Exp(1) by inversion: E = -ln(u). */
double oracle_exp1(uint32_t word)
{
    return -log(oracle_uniform(word));
}

/* ------------------------------------------------------------------------- */
/* Per-row sampling                                                            */
/* ------------------------------------------------------------------------- */
typedef struct {
    float x;
    int32_t idx;
} entry_t;

static int cmp_desc(const void* pa, const void* pb)
{
    const entry_t* a = (const entry_t*)pa;
    const entry_t* b = (const entry_t*)pb;
    if (a->x > b->x) return -1;
    if (a->x < b->x) return 1;
    return (a->idx < b->idx) ? -1 : (a->idx > b->idx);
}

static float read_logit(const void* logits, int dtype, int64_t off)
{
    if (dtype == ORACLE_DTYPE_F32) return ((const float*)logits)[off];
    uint16_t h = ((const uint16_t*)logits)[off];
    uint32_t bits = (uint32_t)h << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

typedef struct {
    /* inputs */
    const void* logits; int dtype; int64_t vocab; int64_t row_stride;
    const int32_t* logit_row;
    const float* temperature; const int32_t* top_k; const float* top_p; const float* min_p;
    const float* presence; const float* frequency; const float* repetition;
    const uint64_t* seed; const uint8_t* has_seed; const uint32_t* stream_id;
    const int32_t* hist_offsets; const int32_t* hist_ids;
    uint64_t global_seed; uint64_t philox_offset;
    const uint32_t* vocab_mask; int64_t mask_stride;
    const int32_t* bias_offsets; const int32_t* bias_ids; const float* bias_values;
    const int32_t* min_tokens_left; const int32_t* stop_offsets; const int32_t* stop_ids;
    int sanitize_nan;
} oracle_in_t;

/* The library's documented per-row limits on logit_bias entries and stop tokens. */
#define ORACLE_MAX_BIAS 64
#define ORACLE_MAX_STOP 16

/* Disallowed tokens of output row r's vocabulary bitmask become -inf: bit
 * (v & 31) of word v >> 5 of the row's mask set means token v is allowed (the
 * grammar's mask applied to the logits before sampling, manual-sglang-101,
 * constrained decoding, step "Mask"). */
static void apply_mask(const oracle_in_t* in, int64_t r, float* x)
{
    if (!in->vocab_mask) return;
    const uint32_t* m = in->vocab_mask + r * in->mask_stride;
    for (int64_t v = 0; v < in->vocab; ++v)
        if (!((m[v >> 5] >> (v & 31)) & 1u)) x[v] = -INFINITY;
}

/* Load output row r's logits as fp32 and apply the penalties for the row's
 * history: count the occurrences c_v of each token, then for c_v > 0
 *   x = x > 0 ? x / rep : x * rep;  x = x - freq * c_v;  x = x - pres,
 * one fp32 operation per step; then the row's vocabulary mask. Returns ST_OK
 * or ST_BAD_HISTORY. */
static int load_penalized_row(const oracle_in_t* in, int64_t r, float* x, int32_t* count,
                              float pres, float freq, float rep)
{
    const int64_t V = in->vocab;
    const int64_t lrow = in->logit_row ? (int64_t)in->logit_row[r] : r;
    for (int64_t v = 0; v < V; ++v) x[v] = read_logit(in->logits, in->dtype, lrow * in->row_stride + v);
    /* NaN sanitising (the manual's SGLANG_SANITIZE_NAN_LOGITS): a NaN logit is -inf */
    if (in->sanitize_nan)
        for (int64_t v = 0; v < V; ++v)
            if (x[v] != x[v]) x[v] = -INFINITY;
    /* logit_bias: each entry adds its value to its token's logit, in list order
     * (one fp32 addition each), before the penalties */
    if (in->bias_offsets) {
        const int32_t b0 = in->bias_offsets[r], b1 = in->bias_offsets[r + 1];
        if (b1 - b0 > ORACLE_MAX_BIAS) return ST_BAD_PARAM;
        for (int32_t j = b0; j < b1; ++j) {
            const int32_t id = in->bias_ids[j];
            if (id < 0 || (int64_t)id >= V) return ST_BAD_PARAM;
        }
        for (int32_t j = b0; j < b1; ++j) x[in->bias_ids[j]] = x[in->bias_ids[j]] + in->bias_values[j];
    }
    /* min_tokens (the first stage of the vLLM sampler the xbrilliance.ai note
     * walks through): while a row still owes tokens, its stop tokens are -inf */
    if (in->stop_offsets) {
        const int32_t s0 = in->stop_offsets[r], s1 = in->stop_offsets[r + 1];
        if (s1 - s0 > ORACLE_MAX_STOP) return ST_BAD_PARAM;
        for (int32_t j = s0; j < s1; ++j)
            if (in->stop_ids[j] < 0 || (int64_t)in->stop_ids[j] >= V) return ST_BAD_PARAM;
        if (in->min_tokens_left && in->min_tokens_left[r] > 0)
            for (int32_t j = s0; j < s1; ++j) x[in->stop_ids[j]] = -INFINITY;
    }
    if (!in->hist_offsets) {
        apply_mask(in, r, x);
        return ST_OK;
    }
    /* the library's documented per-row limit: counts are kept in 16 bits */
    if (in->hist_offsets[r + 1] - in->hist_offsets[r] > 65535) return ST_BAD_HISTORY;
    memset(count, 0, (size_t)V * sizeof(int32_t));
    for (int32_t j = in->hist_offsets[r]; j < in->hist_offsets[r + 1]; ++j) {
        int32_t id = in->hist_ids[j];
        if (id < 0 || (int64_t)id >= V) return ST_BAD_HISTORY;
        count[id] += 1;
    }
    for (int64_t v = 0; v < V; ++v) {
        int32_t c = count[v];
        float xv = x[v];
        if (c > 0) xv = (xv > 0.0f) ? (xv / rep) : (xv * rep);
        float fc = freq * (float)c;
        xv = xv - fc;
        if (c > 0) xv = xv - pres;
        x[v] = xv;
    }
    apply_mask(in, r, x);
    return ST_OK;
}

/* Process output row r. Writes token/status/diag; probs and logprobs (V floats
 * each) when the pointers are non-NULL. Work buffers are caller-provided. */
static void sample_row(const oracle_in_t* in, int64_t r, int32_t* token, int32_t* status,
                       float* probs, float* logprobs, double* diag,
                       float* x, entry_t* order, double* y, int32_t* count, uint8_t* kept)
{
    const int64_t V = in->vocab;
    const float T = in->temperature[r];
    const int32_t k = in->top_k ? in->top_k[r] : -1;
    const float p = in->top_p ? in->top_p[r] : 1.0f;
    const float minp = in->min_p ? in->min_p[r] : 0.0f;
    const float pres = in->presence ? in->presence[r] : 0.0f;
    const float freq = in->frequency ? in->frequency[r] : 0.0f;
    const float rep = in->repetition ? in->repetition[r] : 1.0f;
    const int seeded = in->has_seed ? (in->has_seed[r] != 0) : 0;

    diag[0] = INFINITY; diag[1] = INFINITY; diag[2] = INFINITY; diag[3] = 0.0;
    *token = -1;
    *status = ST_OK;

    /* parameter validation */
    int bad = 0;
    if (!(T >= 0.0f) || isinf(T)) bad = 1;
    if (!(k == -1 || k >= 1)) bad = 1;
    if (!(p > 0.0f && p <= 1.0f)) bad = 1;
    if (!(minp >= 0.0f && minp <= 1.0f)) bad = 1;
    if (!(rep > 0.0f) || isinf(rep)) bad = 1;
    if (!isfinite(pres) || !isfinite(freq)) bad = 1;
    if (bad) { *status = ST_BAD_PARAM; goto fail; }

    /* load the row and apply the penalties */
    {
        int st = load_penalized_row(in, r, x, count, pres, freq, rep);
        if (st != ST_OK) { *status = st; goto fail; }
    }

    /* non-finite checks: NaN or +inf is an error; all -inf is an error */
    int any_finite = 0;
    for (int64_t v = 0; v < V; ++v) {
        if (isnan(x[v]) || (isinf(x[v]) && x[v] > 0)) { *status = ST_NONFINITE; goto fail; }
        if (isfinite(x[v])) any_finite = 1;
    }
    if (!any_finite) { *status = ST_ALL_NEG_INF; goto fail; }

    const int greedy = (T < 1e-5f);
    const double Te = greedy ? 1.0 : (double)T;

    /* greedy pick: argmax of the penalised logits, lowest index on ties */
    int64_t amax = 0;
    for (int64_t v = 1; v < V; ++v) if (x[v] > x[amax]) amax = v;

    for (int64_t v = 0; v < V; ++v) y[v] = (double)x[v] / Te;
    const double ymax = y[amax];

    /* the kept set, stage by stage */
    for (int64_t v = 0; v < V; ++v) kept[v] = 1;
    const int do_topk = (k != -1 && (int64_t)k < V);
    const int do_topp = (p < 1.0f);
    if (do_topk || do_topp) {
        for (int64_t v = 0; v < V; ++v) { order[v].x = x[v]; order[v].idx = (int32_t)v; }
        qsort(order, (size_t)V, sizeof(entry_t), cmp_desc);
        int64_t nk = do_topk ? (int64_t)k : V;
        if (do_topk) for (int64_t i = nk; i < V; ++i) kept[order[i].idx] = 0;
        if (do_topp) {
            /* softmax at T over the top-k set, walked in sorted order */
            double Z = 0.0;
            for (int64_t i = 0; i < nk; ++i) Z += exp(y[order[i].idx] - ymax);
            double S = 0.0;      /* exclusive prefix mass */
            double margin = INFINITY;
            int64_t i = 0;
            for (; i < nk; ++i) {
                double frac = S / Z;
                if (!(frac < (double)p) && i > 0) break;
                double d = fabs(frac - (double)p);
                if (i > 0 && d < margin) margin = d;
                S += exp(y[order[i].idx] - ymax);
            }
            if (i < nk) {
                double d = fabs(S / Z - (double)p);
                if (d < margin) margin = d;
            }
            diag[1] = margin;
            for (int64_t j = i; j < nk; ++j) kept[order[j].idx] = 0;
        }
    }
    if (minp > 0.0f) {
        const double lmin = log((double)minp);
        double margin = INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            if (!kept[v]) continue;
            double rel = y[v] - ymax;
            double d = fabs(rel - lmin);
            if (d < margin) margin = d;
            if (!(rel >= lmin)) kept[v] = 0;
        }
        diag[2] = margin;
    }
    int64_t nkept = 0;
    for (int64_t v = 0; v < V; ++v) nkept += kept[v];
    diag[3] = (double)nkept;

    /* the pick */
    if (greedy) {
        *token = (int32_t)amax;
    } else {
        const uint64_t key = seeded ? in->seed[r] : in->global_seed;
        uint32_t stream = in->stream_id ? in->stream_id[r] : (seeded ? 0u : (uint32_t)r);
        stream = (stream & 0x7FFFFFFFu) | (seeded ? 0x80000000u : 0u);
        double best = -INFINITY, second = -INFINITY;
        int64_t arg = -1;
        for (int64_t v = 0; v < V; ++v) {
            if (!kept[v]) continue;
            uint32_t w = oracle_noise_word(key, stream, in->philox_offset, v);
            double s = y[v] - log(oracle_exp1(w)); /* log(p_v / E_v) up to a constant */
            if (s > best) { second = best; best = s; arg = v; }
            else if (s > second) { second = s; }
        }
        *token = (int32_t)arg;
        diag[0] = best - second;
    }

    /* optional materialisation: softmax / log_softmax over the kept set at T */
    if (probs || logprobs) {
        double Z = 0.0;
        for (int64_t v = 0; v < V; ++v) if (kept[v]) Z += exp(y[v] - ymax);
        const double lse = ymax + log(Z);
        for (int64_t v = 0; v < V; ++v) {
            if (kept[v]) {
                if (probs) probs[v] = (float)exp(y[v] - lse);
                if (logprobs) logprobs[v] = (float)(y[v] - lse);
            } else {
                if (probs) probs[v] = 0.0f;
                if (logprobs) logprobs[v] = -INFINITY;
            }
        }
    }
    return;

fail:
    *token = -1;
    if (probs) for (int64_t v = 0; v < V; ++v) probs[v] = NAN;
    if (logprobs) for (int64_t v = 0; v < V; ++v) logprobs[v] = NAN;
}

/*
 * Sample rows `rows[0..n_out)` (or all n_rows rows when rows == NULL) and write
 * output i for each: out_tokens[i], out_status[i], out_diag[4*i..4*i+3] and, when
 * requested, out_probs / out_logprobs rows i (vocab floats each).
 * diag: [Gumbel top-2 score gap, top-p boundary margin, min-p margin, kept count].
 * Returns 0, or -1 on a missing argument / allocation failure.
 */
int oracle_sample(const void* logits, int dtype, int64_t n_rows, int64_t vocab, int64_t row_stride,
                  const int32_t* logit_row,
                  const float* temperature, const int32_t* top_k, const float* top_p,
                  const float* min_p, const float* presence, const float* frequency,
                  const float* repetition, const uint64_t* seed, const uint8_t* has_seed,
                  const uint32_t* stream_id, const int32_t* hist_offsets, const int32_t* hist_ids,
                  uint64_t global_seed, uint64_t philox_offset,
                  const uint32_t* vocab_mask, int64_t mask_stride,
                  const int32_t* bias_offsets, const int32_t* bias_ids, const float* bias_values,
                  const int32_t* min_tokens_left, const int32_t* stop_offsets, const int32_t* stop_ids,
                  int sanitize_nan,
                  const int64_t* rows, int64_t n_out,
                  int32_t* out_tokens, int32_t* out_status, float* out_probs, float* out_logprobs,
                  double* out_diag, int nthreads)
{
    if (!logits || !temperature || !out_tokens || !out_status || !out_diag || vocab <= 0) return -1;
    if (has_seed && !seed) return -1;
    if (hist_offsets && !hist_ids) return -1;
    oracle_in_t in = {logits, dtype, vocab, row_stride, logit_row, temperature, top_k, top_p, min_p,
                      presence, frequency, repetition, seed, has_seed, stream_id,
                      hist_offsets, hist_ids, global_seed, philox_offset, vocab_mask, mask_stride,
                      bias_offsets, bias_ids, bias_values, min_tokens_left, stop_offsets, stop_ids,
                      sanitize_nan};
    const int64_t n = rows ? n_out : n_rows;
    int failed = 0;
    (void)nthreads;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1) reduction(| : failed)
    {
        float* x = (float*)malloc((size_t)vocab * sizeof(float));
        entry_t* order = (entry_t*)malloc((size_t)vocab * sizeof(entry_t));
        double* y = (double*)malloc((size_t)vocab * sizeof(double));
        int32_t* count = (int32_t*)malloc((size_t)vocab * sizeof(int32_t));
        uint8_t* kept = (uint8_t*)malloc((size_t)vocab);
        const int have_buffers = (x && order && y && count && kept);
        if (!have_buffers) failed = 1;
        /* every thread reaches the work-sharing loop; one without buffers skips its rows */
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n; ++i) {
            if (!have_buffers) { failed = 1; continue; }
            const int64_t r = rows ? rows[i] : i;
            sample_row(&in, r, &out_tokens[i], &out_status[i],
                       out_probs ? out_probs + i * vocab : NULL,
                       out_logprobs ? out_logprobs + i * vocab : NULL,
                       out_diag + 4 * i, x, order, y, count, kept);
        }
        free(x); free(order); free(y); free(count); free(kept);
    }
    return failed ? -1 : 0;
}

/* The penalised (and masked) fp32 logits of output row out_row, whose logits
 * are row `row` of `logits` (the same code the sampler uses), for checking the
 * penalty arithmetic against hand-computed cases. Returns the row status
 * (ST_OK or ST_BAD_HISTORY). */
int oracle_penalized_logits(const void* logits, int dtype, int64_t vocab, int64_t row_stride,
                            int64_t row, float presence, float frequency, float repetition,
                            const int32_t* hist_offsets, const int32_t* hist_ids,
                            const uint32_t* vocab_mask, int64_t mask_stride,
                            const int32_t* bias_offsets, const int32_t* bias_ids, const float* bias_values,
                            const int32_t* min_tokens_left, const int32_t* stop_offsets, const int32_t* stop_ids,
                            int sanitize_nan, int64_t out_row, float* out_x)
{
    oracle_in_t in;
    memset(&in, 0, sizeof in);
    int32_t* lr = (int32_t*)malloc((size_t)(out_row + 1) * sizeof(int32_t));
    int32_t* count = (int32_t*)malloc((size_t)vocab * sizeof(int32_t));
    if (!lr || !count) {
        free(lr);
        free(count);
        return -1;
    }
    lr[out_row] = (int32_t)row;
    in.logits = logits; in.dtype = dtype; in.vocab = vocab; in.row_stride = row_stride;
    in.logit_row = lr;
    in.hist_offsets = hist_offsets; in.hist_ids = hist_ids;
    in.vocab_mask = vocab_mask; in.mask_stride = mask_stride;
    in.bias_offsets = bias_offsets; in.bias_ids = bias_ids; in.bias_values = bias_values;
    in.min_tokens_left = min_tokens_left; in.stop_offsets = stop_offsets; in.stop_ids = stop_ids;
    in.sanitize_nan = sanitize_nan;
    int st = load_penalized_row(&in, out_row, out_x, count, presence, frequency, repetition);
    free(count);
    free(lr);
    return st;
}
