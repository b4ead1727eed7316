/*
 * sampler.h -- C ABI of libsampler.so, the per-decode-step token sampler for
 * GB300 (sm_103a).
 *
 * One call samples one token for each of N output rows of an LLM's [rows, V]
 * logits tensor. Every row carries its own parameters, so one top-p or greedy
 * request never changes what the other rows of the batch compute.
 *
 * The stages, in order, follow the xbrilliance.ai note "采样参数对解码开销的影响：
 * temperature、top_p 与采样核路径" (Effect of sampling parameters on decode cost),
 * section "解码一步里采样做什么" (what sampling does in one decode step):
 *   penalties -> temperature -> top-k / top-p -> min-p -> fp32 softmax and
 *   log_softmax -> pick.
 * The parameters and their defaults follow its section
 * "哪些参数会额外打开一趟全词表计算" (which parameters open an extra full-vocab
 * pass): temperature 1.0, top_p 1.0, top_k -1, min_p 0, presence 0, frequency
 * 0, repetition 1.0. Greedy below T = 1e-5 and the seeded type follow its
 * section "采样类型与选路" (sampling type and routing). The random pick is the
 * Gumbel-max rule of the dev.to claim check "SGLang's +75% sampler speedup
 * skips Qwen3 chat requests", section "Nine lines, and exactly one call site":
 * the token is argmax_v p_v / E_v with E_v ~ Exp(1). Returned logprobs are
 * temperature-scaled, as in the SGLang manual "manual-sglang-101", section
 * "Logprobs are temperature-scaled".
 *
 * Exact semantics (readings of the pages where they are silent):
 *  - penalties, for a token v seen c_v > 0 times in the row's history:
 *        x = x > 0 ? x / repetition : x * repetition;
 *        x = x - frequency * c_v;     x = x - presence;
 *    each step one IEEE fp32 operation, no fused multiply-add;
 *  - T < 1e-5 picks the argmax of the penalised logits (lowest index on ties);
 *    the outputs of such a row use T = 1;
 *  - top_k keeps exactly k tokens in (value desc, index asc) order;
 *    -1 or k >= V keeps all;
 *  - top_p keeps, over the top-k set, the tokens whose exclusive prefix mass
 *    (softmax at T over that set, same order) is < top_p; at least one stays;
 *  - min_p keeps tokens with p_v >= min_p * p_max;
 *  - the pick is argmax over the kept set of x_v / T - ln(E_v), ties to the
 *    lowest index. E_v = -ln(u_v), u_v = (2 * (w >> 9) + 1) * 2^-24, where w is
 *    word (v & 3) of Philox4x32-10 (Salmon et al., SC'11) with
 *        key     = (lo32, hi32) of (has_seed[r] ? seed[r] : global_seed),
 *        counter = (v >> 2, stream, lo32(offset), hi32(offset)),
 *        stream  = (stream_id[r] & 0x7fffffff) | (has_seed[r] ? 0x80000000 : 0);
 *    stream_id == NULL means stream_id[r] = r for unseeded rows and 0 for
 *    seeded rows, so that a seeded row draws the same numbers wherever it sits
 *    in the batch (give the forks of one seeded request distinct stream ids);
 *  - probs = exp(x/T - lse) on the kept set and 0 elsewhere; logprobs =
 *    x/T - lse on the kept set and -inf elsewhere; lse over the kept set.
 *
 * Threading: a handle is used by one host thread and one stream at a time.
 */
#ifndef DECODE_STEP_TOKEN_SAMPLER_H
#define DECODE_STEP_TOKEN_SAMPLER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque handle. */
typedef struct sampler_s* sampler_t;

/* A cudaStream_t (CUstream). NULL is the legacy default stream. */
typedef struct CUstream_st* sampler_stream_t;

/* Logits element types. */
enum {
    SAMPLER_DTYPE_F32 = 0,  /* IEEE binary32 */
    SAMPLER_DTYPE_BF16 = 1  /* bfloat16: the upper 16 bits of a binary32 */
};

/* Return codes of the calls (0 = success; negative = the call did nothing). */
enum {
    SAMPLER_OK = 0,
    SAMPLER_ERR_NULL_ARG = -1,     /* a required pointer is NULL */
    SAMPLER_ERR_BAD_SHAPE = -2,    /* n_rows < 0, vocab < 1, row_stride < vocab, ... */
    SAMPLER_ERR_TOO_LARGE = -3,    /* n_rows > max_rows or vocab > max_vocab */
    SAMPLER_ERR_BAD_DTYPE = -4,
    SAMPLER_ERR_CUDA = -5,         /* a CUDA call failed (launch, copy, set-up) */
    SAMPLER_ERR_NO_DEVICE = -6,    /* no usable sm_100-family device */
    SAMPLER_ERR_NO_STAGING = -7,   /* sampler_sample_host on a handle made without staging */
    SAMPLER_ERR_UNSUPPORTED = -8   /* a feature sampler_sample_noalloc or sampler_sample_ex
                                      does not offer on these arguments */
};

/* Per-row status codes written to out_status (when given). A row with a
 * non-zero status gets token -1 and NaN probs / logprobs; the other rows are
 * unaffected. When several apply, the first in this list is reported. */
enum {
    SAMPLER_ROW_OK = 0,
    SAMPLER_ROW_BAD_PARAM = 3,      /* T < 0, NaN or inf; top_k == 0 or < -1; top_p not
                                       in (0, 1]; min_p not in [0, 1]; repetition <= 0,
                                       NaN or inf; presence / frequency NaN or inf */
    SAMPLER_ROW_BAD_HISTORY = 4,    /* a history id outside [0, V), or more than 65535
                                       ids in one row's history */
    SAMPLER_ROW_NONFINITE = 1,      /* a NaN or +inf logit (after penalties) */
    SAMPLER_ROW_ALL_NEG_INF = 2,    /* every logit is -inf */
    SAMPLER_ROW_TIMEOUT = 5         /* an internal wait gave up (never expected outside
                                       SAMPLER_CREATE_SHORT_WAITS); the call's other rows
                                       and every later call are unaffected */
};

/* Create-time limits. */
typedef struct {
    int device;            /* CUDA device ordinal the handle is bound to */
    int64_t max_rows;      /* largest n_rows a call may pass (>= 1) */
    int64_t max_vocab;     /* largest vocab a call may pass (1 .. 262144) */
    int64_t max_history;   /* sampler_sample_host only: largest total history length */
    uint32_t flags;        /* SAMPLER_CREATE_* bits */
} sampler_config_t;

/* Reserve device staging buffers for sampler_sample_host (max_rows x max_vocab
 * fp32 logits, probs, logprobs, and the per-row arrays). */
#define SAMPLER_CREATE_HOST_STAGING 1u

/* Retired: selected a cluster-per-output-row kernel that has been removed.
 * Accepted and ignored, so that callers built against ABI 1.0 still work. */
#define SAMPLER_CREATE_ROW_KERNEL 2u

/* Test aid: every wait of the small-batch kernel on its own staging copy gives
 * up at once, so each row it samples reports SAMPLER_ROW_TIMEOUT (token -1).
 * The kernel still lets each copy land before it reuses or releases the
 * buffer, so nothing faults and nothing hangs; later calls are unaffected
 * (no state survives a call). Lets a test observe the timeout status. */
#define SAMPLER_CREATE_SHORT_WAITS 4u

/*
 * Arguments of one sampling call. For sampler_sample every pointer is a device
 * pointer; for sampler_sample_host every pointer is a host pointer. The caller
 * owns every buffer. Arrays marked [N] have n_rows entries; NULL optional
 * arrays take the default given.
 */
typedef struct {
    /* logits: rows of `vocab` elements, row i starting at element i * row_stride */
    const void* logits;
    int32_t dtype;                   /* SAMPLER_DTYPE_* */
    int64_t n_rows;                  /* N output rows (0 = nothing to do) */
    int64_t vocab;                   /* V */
    int64_t row_stride;              /* elements between logits rows (>= V) */
    int64_t n_logit_rows;            /* rows in `logits` (only read by sampler_sample_host;
                                        0 = n_rows) */
    const int32_t* logit_row;        /* [N] logits row of output row r (forks share
                                        one); NULL = r */

    const float* temperature;        /* [N] required */
    const int32_t* top_k;            /* [N] NULL = -1 */
    const float* top_p;              /* [N] NULL = 1 */
    const float* min_p;              /* [N] NULL = 0 */
    const float* presence_penalty;   /* [N] NULL = 0 */
    const float* frequency_penalty;  /* [N] NULL = 0 */
    const float* repetition_penalty; /* [N] NULL = 1 */
    const uint64_t* seed;            /* [N] per-row seed, read where has_seed[r] != 0 */
    const uint8_t* has_seed;         /* [N] NULL = no row seeded */
    const uint32_t* stream_id;       /* [N] Philox stream of row r; NULL: see above */

    /* ragged prior-token history, CSR: ids of row r are
       hist_ids[hist_offsets[r] .. hist_offsets[r + 1]); NULL = no penalties */
    const int32_t* hist_offsets;     /* [N + 1] */
    const int32_t* hist_ids;

    uint64_t global_seed;            /* key of unseeded rows */
    uint64_t philox_offset;          /* counter words 2-3 ... */
    const uint64_t* philox_offset_dev; /* ... or read from this device word when non-NULL
                                          (a CUDA graph replays new offsets this way);
                                          ignored by sampler_sample_host */

    int32_t* out_tokens;             /* [N] required */
    float* out_probs;                /* [N * V] row-major, NULL = not materialised */
    float* out_logprobs;             /* [N * V] row-major, NULL = not materialised */
    int32_t* out_status;             /* [N] NULL = not reported */
} sampler_args_t;

/* Create a handle on cfg->device. Returns SAMPLER_OK and sets *out, or a
 * negative code and sets *out = NULL. Allocates device memory only with
 * SAMPLER_CREATE_HOST_STAGING. */
int sampler_create(sampler_t* out, const sampler_config_t* cfg);

/* Enqueue one sampling step on `stream`. All pointers in args are device
 * pointers on the handle's device. Validates only host-visible scalars and
 * pointers, allocates nothing, never synchronizes and never reads device
 * memory on the host; per-row data errors go to out_status. Returns SAMPLER_OK
 * once the work is enqueued, or a negative code (nothing enqueued). The call
 * makes the handle's device current while it runs and restores the caller's
 * current device before returning.
 *
 * Every parameter is per row, so one top-p or greedy request never moves the
 * other rows of the batch to another path: the batch-wide flag problem of the
 * dev.to claim check "SGLang's +75% sampler speedup skips Qwen3 chat
 * requests", section "One request with top_p takes the whole batch off the
 * fast path". The call can be captured in a CUDA graph (no allocation, no
 * synchronization, no host read of device memory, and a Philox offset that may
 * be read from device memory through philox_offset_dev), as the SGLang manual
 * "manual-sglang-101" asks of every step of a captured decode graph in its
 * CUDA-graphs section "The cost: one decode step is a long list of small
 * launches". */
int sampler_sample(sampler_t h, const sampler_args_t* args, sampler_stream_t stream);

/* The same step from host memory: copies the inputs (n_logit_rows rows of
 * logits, the per-row arrays, the history) to the handle's staging buffers on
 * `stream`, samples, copies the outputs back into the host arrays of `args`
 * and synchronizes `stream` before returning. Needs a handle created with
 * SAMPLER_CREATE_HOST_STAGING; history length <= cfg.max_history. Pinned host
 * memory makes the copies asynchronous with respect to other streams. */
int sampler_sample_host(sampler_t h, const sampler_args_t* args, sampler_stream_t stream);

/*
 * Allocation-free sampling step. None of the pages has a counterpart: the
 * sampler they describe always owns its buffers. This entry point takes no
 * handle and allocates nothing. Its workspace (per-row arrival counters and
 * sketch-key histograms, per-(row, slice) records, 3.8 MiB) is an array in the
 * library's own device memory, one copy per device. It runs the same kernel
 * sampler_sample uses for small batches and returns the same tokens. Every
 * launch leaves the counters and histograms at zero, and a row whose wait gave
 * up (SAMPLER_ROW_TIMEOUT) leaves no state behind, so one bad call never
 * affects a later one.
 *
 * The first call on a device does a one-time set-up on the current device:
 * it looks up that array's address, reads the SM count and clears the row
 * counters and histograms on `stream`. Make that first call before any stream capture.
 *
 * Arguments as for sampler_sample (device pointers on the current device),
 * with these limits:
 *   n_rows <= SAMPLER_NOALLOC_MAX_ROWS and vocab <= 262144, else
 *   SAMPLER_ERR_TOO_LARGE;
 *   no history and no out_probs / out_logprobs, else SAMPLER_ERR_UNSUPPORTED.
 * Calls on one device share the workspace: two calls whose kernels can run at
 * the same time (different streams, or different host threads without
 * ordering) race and give wrong tokens. Order them on one stream.
 */
#define SAMPLER_NOALLOC_MAX_ROWS 64
int sampler_sample_noalloc(const sampler_args_t* args, sampler_stream_t stream);

/*
 * Extensions of one step (sampler_sample_ex).
 *
 * Per-row logprob outputs without the [N, V] tensors: the sampled token's
 * logprob and the top_n tokens of the row with theirs. By default these are
 * the logprobs of the distribution the row was sampled from, log_softmax(x / T)
 * over its kept set (T := 1 on greedy rows), as the SGLang manual
 * "manual-sglang-101" says returned logprobs are (section "Logprobs are
 * temperature-scaled"); `unscaled` asks for log_softmax(x) over the whole
 * vocabulary instead (that section's original-logprob switch). x is the row's
 * penalised (and masked) logit. Top-n order: value descending, index
 * ascending; past the tokens the distribution gives any mass, ids are -1 and
 * logprobs -inf. Error rows get NaN logprobs and ids -1. out_top_* are
 * [n_rows * top_n] row-major.
 *
 * Vocabulary bitmask: the grammar mask that the manual's constrained-decoding
 * section applies to the logits before sampling (step "Mask"). Bit (v & 31) of
 * word (v >> 5) of output row r's mask, vocab_mask[r * mask_stride + (v >> 5)],
 * set means token v is allowed; a disallowed token's logit is -inf (after the
 * penalties). A row with no allowed finite logit reports SAMPLER_ROW_ALL_NEG_INF.
 *
 * logit_bias: output row r's entries j in [bias_offsets[r], bias_offsets[r + 1])
 * each add bias_values[j] to the logit of token bias_ids[j] (one fp32
 * addition each, in list order, so a repeated token adds up), before the
 * penalties and the mask. At most SAMPLER_MAX_BIAS entries per row; more, or an
 * id outside [0, vocab), is SAMPLER_ROW_BAD_PARAM. The MLX help text on the
 * manual lists logit_bias among the sampler's inputs without defining it; this
 * is the reading taken.
 *
 * min_tokens: while output row r still owes tokens (min_tokens_left[r] > 0),
 * its stop tokens stop_ids[j], j in [stop_offsets[r], stop_offsets[r + 1]),
 * are -inf (after logit_bias, before the penalties and the mask), so the row
 * cannot end yet. This is the first stage of the sampler's fixed order in the
 * xbrilliance.ai note on sampling cost ("what sampling does in one decode
 * step"); the note names the stage without defining it, and this is the usual
 * reading. At most SAMPLER_MAX_STOP stop tokens per row; more, or an id outside
 * [0, vocab), is SAMPLER_ROW_BAD_PARAM whether or not the row owes tokens.
 * NULL min_tokens_left: no row owes tokens.
 *
 * NaN sanitising (sanitize_nan != 0): a NaN logit reads as -inf, so it is
 * never picked and weighs nothing, instead of failing its row with
 * SAMPLER_ROW_NONFINITE (the manual's SGLANG_SANITIZE_NAN_LOGITS switch, in
 * its MLX help text). +inf stays an error; a row with nothing but NaN and -inf
 * reports SAMPLER_ROW_ALL_NEG_INF.
 *
 * Every pointer is a device pointer on the handle's device.
 */
#define SAMPLER_MAX_TOP_N 16
#define SAMPLER_MAX_BIAS 64
#define SAMPLER_MAX_STOP 16
typedef struct {
    int32_t top_n;                /* 0 .. SAMPLER_MAX_TOP_N */
    int32_t unscaled;             /* 0: log_softmax(x / T) over the kept set; 1: log_softmax(x) */
    float* out_token_logprob;     /* [N] logprob of the sampled token; NULL = not reported */
    int32_t* out_top_ids;         /* [N * top_n] (unused when top_n == 0) */
    float* out_top_logprobs;      /* [N * top_n] */
    const uint32_t* vocab_mask;   /* [N * mask_stride] words; NULL = every token allowed */
    int64_t mask_stride;          /* words between rows' masks, >= ceil(vocab / 32) */
    const int32_t* bias_offsets;  /* [N + 1] CSR offsets of the logit_bias entries; NULL = none */
    const int32_t* bias_ids;      /* [bias_offsets[N]] tokens */
    const float* bias_values;     /* [bias_offsets[N]] values */
    const int32_t* min_tokens_left;  /* [N] tokens each row still owes; NULL = none */
    const int32_t* stop_offsets;  /* [N + 1] CSR offsets of the stop tokens; NULL = none */
    const int32_t* stop_ids;      /* [stop_offsets[N]] tokens */
    int32_t sanitize_nan;         /* 1: NaN logits read as -inf */
} sampler_ext_t;

/* sampler_sample plus the extensions of `ext` (NULL: none). Offered on the
 * small-batch path: at most 256 rows, no history and no materialised probs /
 * logprobs; other calls that ask for an extension return
 * SAMPLER_ERR_UNSUPPORTED with nothing enqueued, as does top_n outside
 * [0, SAMPLER_MAX_TOP_N] or a mask_stride below ceil(vocab / 32). The same
 * capture and device rules as sampler_sample apply. */
int sampler_sample_ex(sampler_t h, const sampler_args_t* args, const sampler_ext_t* ext,
                      sampler_stream_t stream);

/*
 * The LM head and the sampler of one decode step (sampler_lm_head_sample).
 *
 * The xbrilliance.ai note on sampling cost (section "what sampling does in one
 * decode step") has the LM head produce the [num_seqs, vocab_size] logits as
 * matmul(hidden_states, embedding.t()) and pass them to the sampler. This call
 * does both: first, on the tensor cores,
 *     logits[i, v] = bf16(sum_k hidden[i, k] * weight[v, k])   (fp32 sums,
 *                                                             round to nearest even)
 * for i < n_logit_rows (n_rows when 0) into args->logits (bf16, row_stride
 * elements apart), then the step of sampler_sample_ex on those logits. When
 * the small-batch kernel takes the step it is launched as the GEMM's
 * programmatic dependent: its set-up overlaps the GEMM's tail and it waits for
 * the GEMM before it reads the logits. The GEMM's waits are bounded; a CTA
 * whose wait gives up leaves its logits unwritten and counts itself in
 * SAMPLER_STAT_LM_HEAD_TIMEOUTS.
 *
 * hidden: [n_logit_rows, hidden_stride] bf16, one row per logits row; weight:
 * [vocab, weight_stride] bf16, one row per token (an untied LM head or the
 * tied embedding). Both 16-byte aligned, strides multiples of 8 elements and
 * >= hidden_dim, else SAMPLER_ERR_BAD_SHAPE. args->dtype must be
 * SAMPLER_DTYPE_BF16 (SAMPLER_ERR_BAD_DTYPE); at most SAMPLER_LM_HEAD_MAX_ROWS
 * logits rows (SAMPLER_ERR_TOO_LARGE). ext as for sampler_sample_ex.
 */
#define SAMPLER_LM_HEAD_MAX_ROWS 256
typedef struct {
    const void* hidden;       /* [n_logit_rows, hidden_stride] bf16 */
    const void* weight;       /* [vocab, weight_stride] bf16 */
    int64_t hidden_dim;       /* K >= 1 */
    int64_t hidden_stride;    /* elements between hidden rows */
    int64_t weight_stride;    /* elements between weight rows */
} sampler_lm_head_t;

int sampler_lm_head_sample(sampler_t h, const sampler_lm_head_t* lm, const sampler_args_t* args,
                           const sampler_ext_t* ext, sampler_stream_t stream);

/* The LM head alone: logits[i, v] for i < rows, v < vocab, computed as by
 * sampler_lm_head_sample, into `logits` (bf16, logits_stride >= vocab elements
 * apart). rows in [1, SAMPLER_LM_HEAD_MAX_ROWS], vocab <= the handle's
 * max_vocab (SAMPLER_ERR_TOO_LARGE); lm checked as above. */
int sampler_lm_head(sampler_t h, const sampler_lm_head_t* lm, void* logits, int64_t logits_stride, int64_t rows,
                    int64_t vocab, sampler_stream_t stream);

/* Release the handle and its device memory. NULL is a no-op. */
void sampler_destroy(sampler_t h);

/* A static string for a return code or a per-row status code. */
const char* sampler_status_string(int code);

/* Diagnostic counters kept on the device (reading one synchronizes the device):
 *   SAMPLER_STAT_EXACT_ROWS  rows of the small-batch kernel whose kept set its
 *                            per-slice candidate lists could not settle (top-k
 *                            above 128, a top-p cut past the lists, too many
 *                            candidates), finished by its slower exact path.
 *   SAMPLER_STAT_LM_HEAD_TIMEOUTS  CTAs of the LM-head GEMM whose bounded wait
 *                            gave up (their logits were left unwritten).
 * Writes the count to *value and clears it when reset != 0. */
enum { SAMPLER_STAT_EXACT_ROWS = 0, SAMPLER_STAT_LM_HEAD_TIMEOUTS = 1 };
int sampler_get_stat(sampler_t h, int which, uint64_t* value, int reset);

/* ABI version of this header: (major << 16) | minor. */
uint32_t sampler_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_STEP_TOKEN_SAMPLER_H */
