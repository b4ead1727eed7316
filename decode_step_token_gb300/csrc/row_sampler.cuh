// row_sampler.cuh -- the fused per-row token sampler kernel for sm_103a.
//
// One thread-block cluster samples one output row. Its C CTAs each own a
// contiguous slice of the vocabulary, staged once from HBM into shared memory by
// bulk (TMA-engine) copies; every later pass over the row reads shared memory.
// The CTAs exchange per-slice summaries through distributed shared memory, and
// rank 0 (the leader) combines them. Stage order, per row (xbrilliance.ai note on
// sampling cost, section "解码一步里采样做什么"):
//
//   P1  load -> penalties -> row max / argmax / non-finite check; a plain
//       temperature row also takes its Gumbel-max pick in this pass
//   R1  leader: status, max, greedy token, min-p threshold, candidate bound
//   top-k / top-p / min-p selection, one of:
//       candidate path: elements >= a provable lower bound of the kept set are
//         gathered, sorted by (value desc, index asc) and cut in double precision
//       radix path: a cluster-wide 4 x 8-bit radix select on the order-preserving
//         key, by count (top-k) or by exact fixed-point softmax mass (top-p)
//   P3  Gumbel-max over the kept set (when not already picked) and the kept
//       mass for the outputs
//   P4  optional fp32 probs / logprobs over the kept set
//
// Random numbers: Philox4x32-10 (philox.cuh). The pick compares x/T - ln E in
// fp32 to find each thread's two best tokens, and settles the best two of the
// row in double precision, so the winner matches a double-precision evaluation
// unless three tokens sit within fp32 rounding of each other.
#pragma once

#include <cfloat>
#include <climits>
#include <cstdint>

#include "philox.cuh"
#include "ptx.cuh"

namespace dst {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kCandPerCta = 512;
constexpr int kCandTotal = 2048;
constexpr int kChunks = 4;
constexpr uint32_t kMaxPolls = 1u << 24;

enum : int32_t {
    kRowOk = 0,
    kRowNonFinite = 1,
    kRowAllNegInf = 2,
    kRowBadParam = 3,
    kRowBadHistory = 4,
    kRowTimeout = 5,
};

enum : uint32_t {
    kFlagNonFinite = 1u,
    kFlagAnyFinite = 2u,
    kFlagBadHistory = 4u,
    kFlagTimeout = 8u,
};

enum : int32_t { kSelNone = 0, kSelCand = 1, kSelRadix = 2 };

struct KernelParams {
    const void* logits;
    int64_t vocab;
    int64_t row_stride;
    int64_t n_logit_rows;
    const int32_t* logit_row;
    const float* temperature;
    const int32_t* top_k;
    const float* top_p;
    const float* min_p;
    const float* presence;
    const float* frequency;
    const float* repetition;
    const uint64_t* seed;
    const uint8_t* has_seed;
    const uint32_t* stream_id;
    const int32_t* hist_offsets;
    const int32_t* hist_ids;
    uint64_t global_seed;
    uint64_t philox_offset;
    const uint64_t* philox_offset_dev;
    int32_t* out_tokens;
    float* out_probs;
    float* out_logprobs;
    int32_t* out_status;
    int32_t slice_len;  // elements per CTA, a multiple of 8
    // per-row logprob outputs of sampler_sample_ex (slice kernel only)
    float* out_tok_lp;
    int32_t* out_top_ids;
    float* out_top_lp;
    int32_t top_n;
    int32_t lp_unscaled;
    // vocabulary bitmask of sampler_sample_ex (slice kernel only): bit v & 31 of
    // word v >> 5 of row r's mask set = token v allowed
    const uint32_t* vocab_mask;
    int64_t mask_stride;
    // logit_bias of sampler_sample_ex (slice kernel only), CSR by output row
    const int32_t* bias_offsets;
    const int32_t* bias_ids;
    const float* bias_values;
    // min_tokens of sampler_sample_ex (slice kernel only): a row that still owes
    // tokens has its stop tokens (CSR by output row) at -inf
    const int32_t* min_tokens_left;
    const int32_t* stop_offsets;
    const int32_t* stop_ids;
    int32_t sanitize_nan;  // NaN logits read as -inf (slice kernel only)
};

// ------------------------------------------------------------------ records
struct GRec {  // one Gumbel candidate
    float s;        // fp32 score x/T - ln E
    int32_t idx;    // token, INT_MAX when empty
    float x;        // penalised logit
    uint32_t w;     // Philox word
};

struct GTop2 {
    GRec a, b;  // a ranks before b
};

__device__ __forceinline__ GRec grec_empty() { return GRec{-INFINITY, INT_MAX, 0.0f, 0u}; }

__device__ __forceinline__ bool grec_better(const GRec& p, const GRec& q)
{
    return p.s > q.s || (p.s == q.s && p.idx < q.idx);
}

__device__ __forceinline__ void top2_insert(GTop2& t, const GRec& r)
{
    if (grec_better(r, t.a)) {
        t.b = t.a;
        t.a = r;
    } else if (grec_better(r, t.b)) {
        t.b = r;
    }
}

__device__ __forceinline__ GRec grec_shfl(const GRec& r, int src_lane_xor)
{
    GRec o;
    o.s = __shfl_xor_sync(0xffffffffu, r.s, src_lane_xor);
    o.idx = __shfl_xor_sync(0xffffffffu, r.idx, src_lane_xor);
    o.x = __shfl_xor_sync(0xffffffffu, r.x, src_lane_xor);
    o.w = __shfl_xor_sync(0xffffffffu, r.w, src_lane_xor);
    return o;
}

__device__ __forceinline__ void top2_warp_reduce(GTop2& t)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        GRec oa = grec_shfl(t.a, off);
        GRec ob = grec_shfl(t.b, off);
        top2_insert(t, oa);
        top2_insert(t, ob);
    }
}

struct alignas(8) Partial {  // one CTA's summary of its slice, read by the leader
    float mx;
    int32_t amax;
    uint32_t flags;
    uint32_t ncand;
    GRec g0, g1;
    unsigned long long zq;  // fixed-point kept mass, 2^-40 units
    float wmax[kWarps];     // per-warp maxima (lower bounds for top-k)
};

struct alignas(8) RowParams {  // read by every CTA for its own use
    float T, Te, invT;
    int32_t k;
    float p, minp, pres, freq, rep;
    int32_t lrow, hlo, hhi;
    uint32_t stream;
    int32_t status;
    int32_t greedy, do_topk, do_topp, do_minp, want_out, has_hist, plain_single;
    uint32_t key_lo, key_hi, off_lo, off_hi;
};

struct alignas(8) Bcast {  // leader results, written into every CTA of the cluster
    int32_t status;
    int32_t done;
    int32_t token;
    int32_t sel;
    float m;
    float xthr;
    float tau;
    float lnz;  // ln of the kept mass relative to exp((x - m) / T)
    uint32_t bkey;
    int32_t bidx;
    int32_t has_bound;
    uint32_t prefix;
    uint32_t pbits;
    int32_t tie_cta;
    int32_t tie_j;
    int32_t amax;
    unsigned long long w_above;
    unsigned long long target;
};

struct alignas(16) Shared {
    uint64_t mbar[kChunks];
    RowParams rp;
    Bcast bc;
    Partial part;
    float red_f[kWarps];
    int32_t red_i[kWarps];
    uint32_t red_u[kWarps];
    unsigned long long red_z[kWarps];
    GTop2 red_g[kWarps];
    unsigned long long scan_w[kWarps];
    uint32_t ncand;
    int32_t found;
    uint32_t hcnt[256];
    unsigned long long hmass[256];
    float wm_all[kMaxCluster * kWarps];
    unsigned long long cand[kCandPerCta];
    unsigned long long sortbuf[kCandTotal];
};

// ------------------------------------------------------------------ element helpers
template <typename InT>
struct ElemTraits;

template <>
struct ElemTraits<float> {
    static constexpr int kPerVec = 4;
    __device__ static __forceinline__ float get(const uint4& v, int e)
    {
        const uint32_t w = e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
        return __uint_as_float(w);
    }
    __device__ static __forceinline__ float load(const void* base, int64_t i)
    {
        return static_cast<const float*>(base)[i];
    }
};

template <>
struct ElemTraits<uint16_t> {  // bf16 bit patterns
    static constexpr int kPerVec = 8;
    __device__ static __forceinline__ float get(const uint4& v, int e)
    {
        const uint32_t w = (e >> 1) == 0 ? v.x : ((e >> 1) == 1 ? v.y : ((e >> 1) == 2 ? v.z : v.w));
        return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
    __device__ static __forceinline__ float load(const void* base, int64_t i)
    {
        return __uint_as_float(uint32_t(static_cast<const uint16_t*>(base)[i]) << 16);
    }
};

// Order-preserving key of an fp32 value (larger value, larger key; -0 == +0).
__device__ __forceinline__ uint32_t f2key(float x)
{
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ bool in_prefix(uint32_t key, int v, uint32_t bkey, int bidx)
{
    return key > bkey || (key == bkey && v <= bidx);
}

// Candidate sort word: larger = earlier in (value desc, index asc) order.
__device__ __forceinline__ unsigned long long cand_word(uint32_t key, int v)
{
    return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(v));
}

__device__ __forceinline__ uint32_t cand_key(unsigned long long c) { return uint32_t(c >> 32); }
__device__ __forceinline__ int cand_idx(unsigned long long c) { return int(~uint32_t(c)); }

// Penalty for a token seen c > 0 times: one IEEE fp32 operation per step.
__device__ __forceinline__ float penalize(float x, uint32_t c, const RowParams& rp)
{
    x = (x > 0.0f) ? __fdiv_rn(x, rp.rep) : __fmul_rn(x, rp.rep);
    x = __fsub_rn(x, __fmul_rn(rp.freq, __uint2float_rn(c)));
    x = __fsub_rn(x, rp.pres);
    return x;
}

// Softmax mass of a kept token in fixed point (2^-40 units of exp((x - m) / T));
// every finite token weighs at least one unit, -inf weighs nothing.
__device__ __forceinline__ unsigned long long mass_q(float x, float m, float invT)
{
    if (!(x > -INFINITY)) return 0ull;
    const float e = expf((x - m) * invT);
    const unsigned long long q = __float2ull_rn(e * 0x1p40f);
    return q ? q : 1ull;
}

__device__ __forceinline__ uint32_t noise_word(const RowParams& rp, int v)
{
    const uint4 blk = philox4x32_10(make_uint4(uint32_t(v) >> 2, rp.stream, rp.off_lo, rp.off_hi),
                                    PhiloxKey{rp.key_lo, rp.key_hi});
    return lane_of(blk, uint32_t(v) & 3u);
}

// Gumbel score in double, the precision of the final comparison.
__device__ __forceinline__ double gumbel_score_f64(float x, float T, uint32_t w)
{
    return double(x) / double(T) - log(noise_exp1_f64(w));
}

// Pick between the two best fp32 candidates in double precision.
__device__ __forceinline__ int settle_top2(const GTop2& t, float T)
{
    if (t.a.idx == INT_MAX) return -1;
    if (t.b.idx == INT_MAX) return t.a.idx;
    const double sa = gumbel_score_f64(t.a.x, T, t.a.w);
    const double sb = gumbel_score_f64(t.b.x, T, t.b.w);
    if (sa > sb || (sa == sb && t.a.idx < t.b.idx)) return t.a.idx;
    return t.b.idx;
}

struct GumbelAcc {
    GTop2 t;
    float thr;  // skip tokens whose score bound is below this
    uint32_t blk_id;
    uint4 blk;
};

__device__ __forceinline__ void gumbel_init(GumbelAcc& g)
{
    g.t.a = grec_empty();
    g.t.b = grec_empty();
    g.thr = -INFINITY;
    g.blk_id = 0xFFFFFFFFu;
}

__device__ __forceinline__ void gumbel_visit(GumbelAcc& g, const RowParams& rp, int v, float x)
{
    if (!(x > -INFINITY)) return;
    const uint32_t bid = uint32_t(v) >> 2;
    if (bid != g.blk_id) {
        g.blk_id = bid;
        g.blk = philox4x32_10(make_uint4(bid, rp.stream, rp.off_lo, rp.off_hi),
                              PhiloxKey{rp.key_lo, rp.key_hi});
    }
    const uint32_t w = lane_of(g.blk, uint32_t(v) & 3u);
    const float y = x * rp.invT;
    // E >= 1 - u, so the score is at most y - ln(1 - u): a cheap bound first
    if (y - __logf(noise_one_minus_u(w)) < g.thr) return;
    const float s = y - logf(noise_exp1_f32(w));
    const GRec r{s, v, x, w};
    if (grec_better(r, g.t.b)) {
        top2_insert(g.t, r);
        const float s2 = g.t.b.s;
        g.thr = s2 - (1e-4f + 1e-6f * fabsf(s2));
    }
}

// ------------------------------------------------------------------ block reductions
__device__ __forceinline__ void maxidx_merge(float& m, int& i, float om, int oi)
{
    if (om > m || (om == m && oi < i)) {
        m = om;
        i = oi;
    }
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Inclusive suffix scan over the block (value of thread t and all threads after it).
__device__ __forceinline__ unsigned long long block_suffix_scan(unsigned long long v, Shared& sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long s = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_down_sync(0xffffffffu, s, off);
        if (lane + off < 32) s += o;
    }
    if (lane == 0) sh.scan_w[wid] = s;  // warp total
    __syncthreads();
    unsigned long long later = 0;
    for (int w = wid + 1; w < kWarps; ++w) later += sh.scan_w[w];
    __syncthreads();
    return s + later;
}

// Exclusive prefix scan (index order) of small counts; also returns the block total.
__device__ __forceinline__ int block_excl_scan(int v, int& total, Shared& sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int s = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += o;
    }
    if (lane == 31) sh.red_i[wid] = s;
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < wid) before += sh.red_i[w];
        tot += sh.red_i[w];
    }
    __syncthreads();
    total = tot;
    return before + s - v;
}

// ------------------------------------------------------------------ slice access
struct Slice {
    const unsigned char* stage;  // staged bytes; element i at byte hb + i * esize
    const uint16_t* cnt;         // history counts per slice element (penalties)
    int n;                       // elements in the slice
    int hoff;                    // head pad in elements
    int v0;                      // first token of the slice
};

template <typename InT, bool kPen, typename F>
__device__ __forceinline__ void for_each(const Slice& sl, const RowParams& rp, F&& f)
{
    constexpr int EPV = ElemTraits<InT>::kPerVec;
    const int nvec = (sl.hoff + sl.n + EPV - 1) / EPV;
    const uint4* vec = reinterpret_cast<const uint4*>(sl.stage);
    for (int j = threadIdx.x; j < nvec; j += kThreads) {
        const uint4 raw = vec[j];
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const int i = j * EPV + e - sl.hoff;
            if (i < 0 || i >= sl.n) continue;
            float x = ElemTraits<InT>::get(raw, e);
            if (kPen) {
                if (rp.has_hist) {
                    const uint32_t c = sl.cnt[i];
                    if (c) x = penalize(x, c, rp);
                }
            }
            f(sl.v0 + i, x);
        }
    }
}

// ------------------------------------------------------------------ kernel pieces
// Every CTA reads its row's parameters and validates them (same answer everywhere).
__device__ __forceinline__ void read_row_params(const KernelParams& P, int r, RowParams& rp)
{
    const int64_t V = P.vocab;
    rp.T = P.temperature[r];
    rp.k = P.top_k ? P.top_k[r] : -1;
    rp.p = P.top_p ? P.top_p[r] : 1.0f;
    rp.minp = P.min_p ? P.min_p[r] : 0.0f;
    rp.pres = P.presence ? P.presence[r] : 0.0f;
    rp.freq = P.frequency ? P.frequency[r] : 0.0f;
    rp.rep = P.repetition ? P.repetition[r] : 1.0f;
    const bool seeded = P.has_seed ? (P.has_seed[r] != 0) : false;
    const uint64_t key = seeded ? P.seed[r] : P.global_seed;
    uint32_t stream = P.stream_id ? P.stream_id[r] : (seeded ? 0u : uint32_t(r));
    rp.stream = (stream & 0x7FFFFFFFu) | (seeded ? 0x80000000u : 0u);
    rp.key_lo = uint32_t(key);
    rp.key_hi = uint32_t(key >> 32);
    const uint64_t off = P.philox_offset_dev ? *P.philox_offset_dev : P.philox_offset;
    rp.off_lo = uint32_t(off);
    rp.off_hi = uint32_t(off >> 32);
    rp.lrow = P.logit_row ? P.logit_row[r] : r;
    rp.has_hist = P.hist_offsets != nullptr;
    rp.hlo = rp.has_hist ? P.hist_offsets[r] : 0;
    rp.hhi = rp.has_hist ? P.hist_offsets[r + 1] : 0;

    bool bad = false;
    if (!(rp.T >= 0.0f) || isinf(rp.T)) bad = true;
    if (!(rp.k == -1 || rp.k >= 1)) bad = true;
    if (!(rp.p > 0.0f && rp.p <= 1.0f)) bad = true;
    if (!(rp.minp >= 0.0f && rp.minp <= 1.0f)) bad = true;
    if (!(rp.rep > 0.0f) || isinf(rp.rep)) bad = true;
    if (!isfinite(rp.pres) || !isfinite(rp.freq)) bad = true;
    rp.status = bad ? kRowBadParam : kRowOk;

    rp.greedy = rp.T < 1e-5f;
    rp.Te = rp.greedy ? 1.0f : rp.T;
    rp.invT = 1.0f / rp.Te;
    rp.do_topk = (rp.k != -1 && int64_t(rp.k) < V);
    rp.do_topp = rp.p < 1.0f;
    rp.do_minp = rp.minp > 0.0f;
    rp.want_out = (P.out_probs != nullptr) || (P.out_logprobs != nullptr);
    rp.plain_single = !rp.greedy && !rp.do_topk && !rp.do_topp && !rp.do_minp && !rp.want_out;
}

}  // namespace dst
