// slice_kernel.cuh -- body of the slice kernel (design in slice_sampler.cuh).
//
// Every warp runs on its own: its unit's copy, its row's parameters, its
// summary, its arrival and, when it completes a row, that row's finish. The
// only CTA-wide step is the exact path at the end, for rows the candidate
// lists could not settle.
//
// Included once per kernel variant, into namespace SLC_VARIANT: SLC_FILTERS 1
// takes the filters of sampler_sample_ex (vocabulary mask, logit_bias,
// min_tokens, NaN sanitising), SLC_LP 1 its logprob outputs; 0 compiles that
// code out. The plain step's variant (both 0) has about half the kernel text of
// the one with everything (its finishing code runs from a cold instruction
// cache, so the text it walks through is what it pays for).
#if !defined(SLC_FILTERS) || !defined(SLC_LP) || !defined(SLC_VARIANT)
#error "define SLC_FILTERS, SLC_LP (0 or 1) and SLC_VARIANT before including slice_kernel.cuh"
#endif

#include "slice_sampler.cuh"

// Timeline hooks: a profiling build defines them to record a timestamp per warp
// and event; they compile to nothing otherwise.
#ifndef SLC_MARK
#define SLC_MARK(i)
#define SLC_TAG(v)
#define SLC_UCLS(v)
#endif
#ifndef SLC_FIN_INLINE
#define SLC_FIN_INLINE __forceinline__
#endif

namespace dst {
namespace slc {
namespace SLC_VARIANT {

// ---------------------------------------------------------------- extension switches
// Constant false in the variants without them, so that their code drops out.
__device__ __forceinline__ bool row_lp(const RowInfo& ri) { return SLC_LP && ri.lp; }
__device__ __forceinline__ const uint32_t* mask_of(const KernelParams& kp)
{
    return SLC_FILTERS ? kp.vocab_mask : nullptr;
}
__device__ __forceinline__ bool sanitizing(const KernelParams& kp) { return SLC_FILTERS && kp.sanitize_nan; }

// ---------------------------------------------------------------- set-up
// Every lane of the warp reads the same row (one request each, the same words).
__device__ __forceinline__ RowInfo load_info(const SliceParams& P, int r)
{
    const KernelParams& kp = P.k;
    const int64_t V = kp.vocab;
    RowInfo ri;
    const float T = kp.temperature[r];
    ri.k = kp.top_k ? kp.top_k[r] : -1;
    ri.p = kp.top_p ? kp.top_p[r] : 1.0f;
    ri.minp = kp.min_p ? kp.min_p[r] : 0.0f;
    const float pres = kp.presence ? kp.presence[r] : 0.0f;
    const float freq = kp.frequency ? kp.frequency[r] : 0.0f;
    const float rep = kp.repetition ? kp.repetition[r] : 1.0f;
    const bool seeded = kp.has_seed ? kp.has_seed[r] != 0 : false;
    const uint64_t key = seeded ? kp.seed[r] : kp.global_seed;
    const uint32_t sid = kp.stream_id ? kp.stream_id[r] : (seeded ? 0u : uint32_t(r));
    const int lrow = kp.logit_row ? kp.logit_row[r] : r;
    ri.stream = (sid & 0x7FFFFFFFu) | (seeded ? 0x80000000u : 0u);
    ri.key_lo = uint32_t(key);
    ri.key_hi = uint32_t(key >> 32);
    ri.lrow = lrow < 0 ? 0 : lrow;
    bool bad = lrow < 0;
    if (!(T >= 0.0f) || isinf(T)) bad = true;
    if (!(ri.k == -1 || ri.k >= 1)) bad = true;
    if (!(ri.p > 0.0f && ri.p <= 1.0f)) bad = true;
    if (!(ri.minp >= 0.0f && ri.minp <= 1.0f)) bad = true;
    if (!isfinite(pres) || !isfinite(freq)) bad = true;
    if (!(rep > 0.0f) || isinf(rep)) bad = true;
    // min_tokens: the row's stop tokens are banned while it owes tokens (the
    // lists' limits are checked warp-wide by ext_lists_ok)
    ri.ban = 0;
    if (SLC_FILTERS && kp.stop_offsets && kp.min_tokens_left && kp.min_tokens_left[r] > 0 &&
        kp.stop_offsets[r + 1] > kp.stop_offsets[r])
        ri.ban = 1;
    const bool greedy = T < 1e-5f;
    ri.T = greedy ? 1.0f : T;
    ri.invT = 1.0f / ri.T;
    ri.s2 = 1.4426950408889634f / ri.T;
    ri.do_topk = (ri.k != -1 && int64_t(ri.k) < V);
    ri.do_topp = ri.p < 1.0f;
    ri.do_minp = ri.minp > 0.0f;
    ri.need_z = ri.do_topp && !ri.do_topk;
    ri.m = uint8_t(ri.do_topk ? min(ri.k, kSketch) : kSketch);
    // the list threshold: the k-th largest lane maximum on a top-k row with
    // k <= kKComplete (the list then holds the unit's top k), else the m-th
    ri.mt = uint8_t(ri.do_topk && ri.k <= kKComplete ? ri.k : ri.m);
    ri.greedy = greedy ? 1 : 0;
    const bool trunc = ri.do_topk || ri.do_topp || ri.do_minp;
    ri.lp = (SLC_LP && (kp.out_tok_lp != nullptr || kp.top_n > 0)) ? 1 : 0;
    if (bad) ri.cls = kClsErr;
    else if (greedy) ri.cls = (ri.lp && trunc) ? kClsTrunc : kClsGreedy;  // outputs over the kept set at T := 1
    else if (!trunc) ri.cls = kClsPlain;
    else ri.cls = kClsTrunc;
    // the logprob outputs: over the kept set at T (scaled, truncated rows: from
    // the finisher's candidates), else over the whole row at T_out, from masses
    // the units keep; every unit lists at least its top n
    ri.s2o = kp.lp_unscaled ? 1.4426950408889634f : ri.s2;
    ri.need_zo = (ri.lp && (kp.lp_unscaled || ri.cls != kClsTrunc)) ? 1 : 0;
    if (ri.lp && kp.top_n > 0) ri.mt = uint8_t(max(int(ri.mt), kp.top_n));
    ri.pad3 = 0;
    ri.r = r;
    return ri;
}

// First element of the slice starting at token c0 of logits row lrow.
template <typename InT>
__device__ __forceinline__ const InT* slice_ptr(const KernelParams& kp, int lrow, int c0)
{
    return static_cast<const InT*>(kp.logits) + (int64_t(lrow) * kp.row_stride + c0);
}

// Whole 16-byte vectors of a slice that the bulk copy moves (0 when the slice
// does not start on a 16-byte boundary).
template <typename InT>
__device__ __forceinline__ int bulk_vecs(const InT* g, int n)
{
    if ((reinterpret_cast<uintptr_t>(g) & 15u) != 0) return 0;
    return int((size_t(n) * sizeof(InT)) / 16);
}

// Lane 0: arm the warp's mbarrier for its next phase and start the unit's copy.
template <typename InT>
__device__ __forceinline__ void issue_unit(const SliceParams& P, uint64_t* bar, unsigned char* slot, int u)
{
    const KernelParams& kp = P.k;
    const int r = u / P.G, s = u - r * P.G;
    int lrow = kp.logit_row ? kp.logit_row[r] : r;
    lrow = lrow < 0 ? 0 : lrow;
    const int c0 = s * P.W;
    const int n = min(P.W, int(kp.vocab) - c0);
    const InT* g = slice_ptr<InT>(kp, lrow, c0);
    const uint32_t bytes = uint32_t(bulk_vecs<InT>(g, n)) * 16u;
    mbar_arrive_expect_tx(bar, bytes);
    if (bytes) bulk_copy_g2s(slot, g, bytes, bar);
}

// Atomic add with release and acquire semantics at GPU scope.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t philox_word(const RowPhilox& rp, int v)
{
    return lane_of(philox_block(rp, uint32_t(v) >> 2), uint32_t(v) & 3u);
}

// First position of value m in a vector that holds it.
template <typename InT>
__device__ __forceinline__ int vec_find(const uint4& v, float m)
{
    constexpr int E = Vec<InT>::E;
    int pos = E - 1;
#pragma unroll
    for (int e = E - 1; e >= 0; --e)
        if (Vec<InT>::get(v, e) == m) pos = e;
    return pos;
}

// NaN sanitising of the vectors a lane reads (the unit is staged whole): NaN
// becomes -inf in the slot; returns the lane's new maximum.
template <typename InT>
__device__ __noinline__ float lane_sanitize(SliceView<InT> sv)
{
    const int lane = threadIdx.x & 31;
    uint4* smv = const_cast<uint4*>(sv.sm);
    typename Vec<InT>::Acc a = Vec<InT>::acc_init();
#pragma unroll 1
    for (int j = lane; j < sv.nvec; j += 32) {
        const uint4 c = Vec<InT>::sanitized(smv[j]);
        smv[j] = c;
        Vec<InT>::acc_add(a, c);
    }
    return Vec<InT>::acc_max(a);
}

// Lane maximum and the flags of the part of the unit a lane reads: one packed,
// NaN-propagating maximum per vector. A lane that met a NaN reports -inf (its
// flags mark the row).
template <typename InT>
__device__ __forceinline__ float lane_max_val(const SliceView<InT>& sv, uint32_t& f)
{
    const int lane = threadIdx.x & 31;
    typename Vec<InT>::Acc a = Vec<InT>::acc_init();
#pragma unroll 2
    for (int j = lane; j < sv.nvec; j += 32) Vec<InT>::acc_add(a, sv.vec(j));
    float m = Vec<InT>::acc_max(a);
    if (SLC_FILTERS && sv.san) {
        // NaN sanitising (the unit is staged whole): a lane that met a NaN makes
        // its NaNs -inf in the slot and takes its maximum again
        if (m != m) m = lane_sanitize<InT>(sv);
        __syncwarp();
    }
    const bool nan = m != m;
    f = flags_of(nan, m);
    return nan ? -INFINITY : m;
}

// Lowest token of the lane's part of the unit equal to m (a value the lane holds).
template <typename InT>
__device__ __forceinline__ int lane_find(const SliceView<InT>& sv, float m)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int j = lane; j < sv.nvec; j += 32) {
        const uint4 v = sv.vec(j);
        if (Vec<InT>::has(v, m)) return sv.c0 + j * E + vec_find<InT>(v, m);
    }
    return INT_MAX;
}

// Lane maximum, its lowest token (INT_MAX when nothing is finite) and flags.
template <typename InT>
__device__ __forceinline__ void lane_max(const SliceView<InT>& sv, float& m, int& mi, uint32_t& f)
{
    m = lane_max_val<InT>(sv, f);
    mi = m > -INFINITY ? lane_find<InT>(sv, m) : INT_MAX;
}

// Unit maximum and its lowest token (only lanes holding the maximum search);
// lm gets the lane maximum.
template <typename InT>
__device__ __forceinline__ void unit_max(const SliceView<InT>& sv, float& mx, int& amax, uint32_t& flags, float& lm)
{
    uint32_t f;
    lm = lane_max_val<InT>(sv, f);
    flags = warp_or(f);
    mx = key2f(__reduce_max_sync(0xffffffffu, f2key(lm)));
    int li = INT_MAX;
    if (mx > -INFINITY && lm == mx) li = lane_find<InT>(sv, lm);
    amax = __reduce_min_sync(0xffffffffu, li);
}

// ---------------------------------------------------------------- logit_bias, min_tokens
// Whether the row carries logit_bias or stop-token lists (row_extras checks
// them and takes the biased and banned tokens apart from the staged logits).
__device__ __forceinline__ bool has_extras(const KernelParams& kp)
{
    return SLC_FILTERS && (kp.bias_offsets != nullptr || kp.stop_offsets != nullptr);
}

// Row r's logit of token v after NaN sanitising, its bias entries (one fp32
// addition each, in list order), its min_tokens ban and its vocabulary mask:
// one thread's view, for the few tokens read again one by one.
template <typename InT>
__device__ __forceinline__ float biased_logit(const KernelParams& kp, const RowInfo& ri, int v)
{
    float x = ElemTraits<InT>::load(kp.logits, int64_t(ri.lrow) * kp.row_stride + v);
    if (sanitizing(kp) && x != x) x = -INFINITY;
    if (mask_of(kp) && !((__ldg(mask_of(kp) + size_t(ri.r) * size_t(kp.mask_stride) + (v >> 5)) >> (v & 31)) & 1u))
        return -INFINITY;
    if (SLC_FILTERS && ri.ban) {
        const int s1 = kp.stop_offsets[ri.r + 1];
        for (int j = kp.stop_offsets[ri.r]; j < s1; ++j)
            if (kp.stop_ids[j] == v) return -INFINITY;
    }
    if (SLC_FILTERS && kp.bias_offsets) {
        const int b1 = kp.bias_offsets[ri.r + 1];
        for (int j = kp.bias_offsets[ri.r]; j < b1; ++j)
            if (kp.bias_ids[j] == v) x = x + kp.bias_values[j];
    }
    return x;
}

// The row's biased and banned tokens in [lo, hi) with their final logits (each
// token once), written to xi / xv; returns how many (at most kMaxExtras), or
// -1 when the row's lists break the limits (more than kMaxBias / kMaxStop
// entries, an id outside the vocabulary). Warp-wide.
template <typename InT>
__device__ __noinline__ int row_extras(const KernelParams& kp, RowInfo ri, int lo, int hi, int32_t* xi,
                                       float* xv)
{
    constexpr int K = (kMaxExtras + 31) / 32;  // entries per lane
    const int lane = threadIdx.x & 31;
    const int64_t V = kp.vocab;
    const int b0 = kp.bias_offsets ? kp.bias_offsets[ri.r] : 0;
    const int Lb = kp.bias_offsets ? kp.bias_offsets[ri.r + 1] - b0 : 0;
    const int s0 = kp.stop_offsets ? kp.stop_offsets[ri.r] : 0;
    const int Ls = kp.stop_offsets ? kp.stop_offsets[ri.r + 1] - s0 : 0;
    if (Lb < 0 || Lb > kMaxBias || Ls < 0 || Ls > kMaxStop) return -1;
    const int L = Lb + Ls;
    // Lane l holds entries l, l + 32, ... of the bias list followed by the stop
    // tokens, and for those in [lo, hi) the token's logit and mask bit: every
    // load is issued before any is used.
    int id[K];
    float bv[K], x[K];
    bool ok[K];
    bool bad = false;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int e = lane + 32 * k;
        id[k] = e < Lb ? kp.bias_ids[b0 + e] : e < L ? kp.stop_ids[s0 + (e - Lb)] : -1;
        bv[k] = e < Lb ? kp.bias_values[b0 + e] : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int e = lane + 32 * k;
        bad |= e < L && (id[k] < 0 || int64_t(id[k]) >= V);
        if (e >= Lb && !ri.ban) id[k] = -1;  // stop tokens ban nothing once the row owes none
    }
    if (__any_sync(0xffffffffu, bad)) return -1;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const bool in = id[k] >= lo && id[k] < hi;
        x[k] = in ? ElemTraits<InT>::load(kp.logits, int64_t(ri.lrow) * kp.row_stride + id[k]) : 0.0f;
        ok[k] = !in || !mask_of(kp) ||
                ((__ldg(mask_of(kp) + size_t(ri.r) * size_t(kp.mask_stride) + (id[k] >> 5)) >> (id[k] & 31)) & 1u);
    }
    // the tokens in range, each at its first entry, in list order
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        uint32_t todo = __ballot_sync(0xffffffffu, id[k] >= lo && id[k] < hi);
#pragma unroll 1
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1u;
            const int v = __shfl_sync(0xffffffffu, id[k], src);
            uint32_t mt[K];
            bool first = true;
#pragma unroll
            for (int kk = 0; kk < K; ++kk) {
                mt[kk] = __ballot_sync(0xffffffffu, id[kk] == v);
                if (kk < k && mt[kk]) first = false;
            }
            if (mt[k] & ((1u << src) - 1u)) first = false;
            if (!first) continue;
            // the token's value: its logit plus its bias entries in list order;
            // -inf when a stop-token entry bans it or its mask bit is clear
            float acc = __shfl_sync(0xffffffffu, x[k], src);
            if (sanitizing(kp) && acc != acc) acc = -INFINITY;
            bool banned = !__shfl_sync(0xffffffffu, ok[k], src);
#pragma unroll
            for (int kk = 0; kk < K; ++kk) {
#pragma unroll 1
                for (uint32_t m = mt[kk]; m; m &= m - 1u) {
                    const int j = __ffs(m) - 1;
                    const float b = __shfl_sync(0xffffffffu, bv[kk], j);
                    if (j + 32 * kk < Lb) acc = acc + b;
                    else banned = true;
                }
            }
            if (lane == 0) {
                xi[cnt] = v;
                xv[cnt] = banned ? -INFINITY : acc;
            }
            ++cnt;
        }
    }
    __syncwarp();
    return cnt;
}

// Whether token v is among the n biased tokens xi.
__device__ __forceinline__ bool is_extra(const int32_t* xi, int n, int v)
{
    for (int q = 0; q < n; ++q)
        if (xi[q] == v) return true;
    return false;
}

// Flags of the extras' values (NaN or +inf: non-finite; finite: any finite).
__device__ __forceinline__ uint32_t extras_flags(const float* xv, int n)
{
    const int lane = threadIdx.x & 31;
    uint32_t f = 0;
    for (int q = lane; q < n; q += 32) {
        const float x = xv[q];
        if (x != x || x == INFINITY) f |= kFlagNonFinite;
        if (x > -INFINITY && x < INFINITY) f |= kFlagAnyFinite;
    }
    return warp_or(f);
}

// Merge the extras into a unit maximum (value desc, index asc; NaN ignored).
__device__ __forceinline__ void extras_max(const int32_t* xi, const float* xv, int n, float& mx, int& amax)
{
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
    int mi = INT_MAX;
    for (int q = lane; q < n; q += 32) {
        const float x = xv[q];
        if (x > m || (x == m && xi[q] < mi)) {
            m = x;
            mi = xi[q];
        }
    }
    warp_max_idx(m, mi);
    if (m > mx || (m == mx && mi < amax)) {
        mx = m;
        amax = mi;
    }
}

// ---------------------------------------------------------------- plain unit
// Philox words of the 8 (bf16) or 4 (fp32) tokens of the vector starting at t0:
// for bf16 two independent blocks computed side by side.
template <typename InT>
__device__ __forceinline__ void vec_words(const RowPhilox& rp, int t0, uint4& b0, uint4& b1)
{
    if constexpr (Vec<InT>::E == 8) {
        constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
        const uint32_t c0 = uint32_t(t0) >> 2, c1 = c0 + 1u;
        uint32_t ha0, la0, hb0, lb0, ha1, la1, hb1, lb1;
        mul_wide(kMulA, c0, ha0, la0);
        mul_wide(kMulA, c1, ha1, la1);
        mul_wide(kMulB, ha0 ^ rp.r1z, hb0, lb0);
        mul_wide(kMulB, ha1 ^ rp.r1z, hb1, lb1);
        uint32_t x0 = hb0 ^ rp.r2x, y0 = lb0, z0 = rp.r2z ^ la0, w0 = rp.r2w;
        uint32_t x1 = hb1 ^ rp.r2x, y1 = lb1, z1 = rp.r2z ^ la1, w1 = rp.r2w;
#pragma unroll
        for (int round = 2; round < 10; ++round) {
            mul_wide(kMulA, x0, ha0, la0);
            mul_wide(kMulA, x1, ha1, la1);
            mul_wide(kMulB, z0, hb0, lb0);
            mul_wide(kMulB, z1, hb1, lb1);
            x0 = hb0 ^ y0 ^ rp.k0[round];
            z0 = ha0 ^ w0 ^ rp.k1[round];
            x1 = hb1 ^ y1 ^ rp.k0[round];
            z1 = ha1 ^ w1 ^ rp.k1[round];
            y0 = lb0;
            w0 = la0;
            y1 = lb1;
            w1 = la1;
        }
        b0 = make_uint4(x0, y0, z0, w0);
        b1 = make_uint4(x1, y1, z1, w1);
    } else {
        b0 = philox_block(rp, uint32_t(t0) >> 2);
        b1 = b0;
    }
}

// Cheap test against the threshold thr (log2 units) of the bound
// x s2 - log2(1 - u): lets through every token the bound keeps. With
// L = a 2^-23 <= 1 - u (a = the word's top 23 bits complemented) and the bit
// pattern of L read as a number (at most log2 L, plus 127, in 2^-23 units), the
// test is bits(L) <= (x s2 - thr + 127) 2^23, evaluated in 2^-16 units on
// floats. Negative result = let through.
struct CheapBound {
    float A, K;
    __device__ __forceinline__ CheapBound(float s2, float thr)
    {
        A = s2 * 65536.0f;
        // K = 2^23 + (127 - thr + eps) 2^16 + 4, rounded up; eps covers the fp32
        // bound's own rounding
        const double eps = 2e-3 + 1e-6 * fabs(double(thr));
        K = __double2float_ru(8388608.0 + (127.0 - double(thr) + eps) * 65536.0 + 4.0);
    }
    __device__ __forceinline__ float d(float x, uint32_t w) const
    {
        const float g = __uint_as_float(0x3F800000u + (w >> 9));  // 1 + (w >> 9) 2^-23
        const float L = 1.99999988079071044921875f - g;            // (2 - 2^-23) - g = a 2^-23, exact
        const float F = __uint_as_float(0x4B000000u + (__float_as_uint(L) >> 7));
        return F - fmaf(x, A, K);
    }
};

template <typename InT>
__device__ __forceinline__ void unit_plain(const SliceView<InT>& sv, const RowInfo& ri, uint32_t off_lo,
                                           uint32_t off_hi, uint16_t* q, uint4* qw, K2& out, uint32_t& flags)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    // each lane scores its largest logit exactly; the second-best of these 32
    // scores bounds the unit's second-best score from below
    float lm;
    int li;
    uint32_t f;
    lane_max<InT>(sv, lm, li, f);
    SLC_MARK(4);
    flags = warp_or(f);
    const RowPhilox rp = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, off_lo, off_hi);
    const float s2 = ri.s2;
    K2 t{0ull, 0ull};
    uint32_t sk = 0;
    if (lm > -INFINITY && lm < INFINITY) {
        const float ss = score2(lm, s2, philox_word(rp, li));
        t.a = gkey(ss, li);
        sk = f2key(ss);
    }
    const uint32_t k1 = __reduce_max_sync(0xffffffffu, sk);
    const uint32_t holder = __ballot_sync(0xffffffffu, sk == k1);
    const uint32_t k2 = __reduce_max_sync(0xffffffffu, lane == __ffs(holder) - 1 ? 0u : sk);
    float thr = -INFINITY;
    if (k2 != 0) {
        thr = key2f(k2);
        thr -= 1e-4f + 4e-6f * fabsf(thr);
    }
    // pass 1: the cheap test over every token; vectors with a token through are
    // queued (warp-private, in order; the first 32 with their Philox words), so
    // that the exact scoring below runs with all lanes busy
    const CheapBound cb(s2, thr);
    int nq = 0;
    SLC_MARK(20);
    // two vectors' Philox blocks overlap (measured faster than one at a time)
#pragma unroll 2
    for (int j0 = 0; j0 < sv.nvec; j0 += 32) {
        const int j = j0 + lane;
        uint32_t neg = 0;
        uint4 b0, b1;
        if (j < sv.nvec) {
            const uint4 v = sv.vec(j);
            vec_words<InT>(rp, sv.c0 + j * E, b0, b1);
#pragma unroll
            for (int e = 0; e < E; ++e)
                neg |= __float_as_uint(cb.d(Vec<InT>::get(v, e), lane_of(e < 4 ? b0 : b1, uint32_t(e) & 3u)));
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, (neg >> 31) != 0u);
        if (neg >> 31) {
            const int at = nq + __popc(bal & ((1u << lane) - 1u));
            q[at] = uint16_t(j);
            if (at < 32) {
                qw[2 * at] = b0;
                qw[2 * at + 1] = b1;
            }
        }
        nq += __popc(bal);
    }
    __syncwarp();
    SLC_MARK(21);
    // pass 2: exact scores of the queued vectors' tokens that pass the test; a
    // vector may go to another lane than the one that read it, whose largest
    // logit (already scored) is skipped
#pragma unroll 1
    for (int i0 = 0; i0 < nq; i0 += 32) {
        const int i = i0 + lane;
        const int j = i < nq ? int(q[i]) : 0;
        const int oli = __shfl_sync(0xffffffffu, li, j & 31);
        if (i < nq) {
            const uint4 v = sv.vec(j);
            const int t0 = sv.c0 + j * E;
            uint4 b0, b1;
            if (i < 32) {
                b0 = qw[2 * i];
                b1 = qw[2 * i + 1];
            } else {
                vec_words<InT>(rp, t0, b0, b1);
            }
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float x = Vec<InT>::get(v, e);
                const uint32_t we = lane_of(e < 4 ? b0 : b1, uint32_t(e) & 3u);
                if (t0 + e == oli || !(x > -INFINITY) || !(cb.d(x, we) < 0.0f)) continue;
                k2_insert(t, gkey(score2(x, s2, we), t0 + e));
            }
        }
    }
    __syncwarp();
    k2_warp_reduce(t);
    out = t;
}

// ---------------------------------------------------------------- truncated unit
// Position of the n-th set bit (counting from 0) of a mask that has more than n.
__device__ __forceinline__ int nth_set_lane(uint32_t mask, int n)
{
    int pos = 0;
#pragma unroll
    for (int w = 16; w > 0; w >>= 1)
        if (__popc(mask & ((1u << (pos + w)) - 1u)) <= n) pos += w;
    return pos;
}

// Bin of a sketch key in its row's histogram: 1/4 wide over the logits
// [-32, 32), the outer two bins taking everything beyond.
__device__ __forceinline__ uint32_t key_bin(uint32_t key)
{
    const int b = __float2int_rd(key2f(key) * 4.0f) + kHistBins / 2;
    return uint32_t(min(max(b, 0), kHistBins - 1));
}

// 16-bit prefixes that enclose bin b: every key of the bin reaches lo << 16,
// and a key that reaches hi << 16 lies in a higher bin (inner bins only).
__device__ __forceinline__ uint32_t bin_lo_prefix(int b)
{
    return f2key(float(b - kHistBins / 2) * 0.25f) >> 16;
}
__device__ __forceinline__ uint32_t bin_hi_prefix(int b)
{
    return (f2key(float(b + 1 - kHistBins / 2) * 0.25f) >> 16) + 1u;
}

// Sum over the unit of exp2((x - mx) * s2) (Kahan per lane, double across the
// warp), as a high and a low fp32 part.
template <typename InT>
__device__ __noinline__ void unit_mass(SliceView<InT> sv, float mx, float s2, float& hi, float& lo,
                                       const float* xv = nullptr, int nx = 0)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    float zs = 0.0f, zc = 0.0f;  // Kahan: the sum is zs - zc
#pragma unroll 1
    for (int j = lane; j < sv.nvec; j += 32) {
        const uint4 v = sv.vec(j);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float x = Vec<InT>::get(v, e);
            if (!(x > -INFINITY)) continue;
            const float term = exp2f((x - mx) * s2) - zc;
            const float sum = zs + term;
            zc = (sum - zs) - term;
            zs = sum;
        }
    }
    double z = double(zs) - double(zc);
    for (int q = lane; q < nx; q += 32)  // biased tokens (read as -inf above)
        if (xv[q] > -INFINITY) z += double(exp2f((xv[q] - mx) * s2));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    hi = float(z);
    lo = float(z - double(hi));
}

template <typename InT>
__device__ __forceinline__ void unit_trunc(const SliceView<InT>& sv, const RowInfo& ri, SliceHdr& hdr_out,
                                           SliceBody* body, uint32_t* q, const int32_t* xi = nullptr,
                                           const float* xv = nullptr, int nx = 0, uint32_t* hist = nullptr)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    float lm, mx;
    int amax;
    uint32_t flags;
    unit_max<InT>(sv, mx, amax, flags, lm);
    // biased tokens (read as -inf by sv) count in the maximum, the flags, the
    // list and the mass, not in the lane maxima: the sketch and tau keep their
    // meaning (tokens of the unit that reach them)
    if (nx) {
        flags |= extras_flags(xv, nx);
        extras_max(xi, xv, nx, mx, amax);
    }
    SLC_MARK(4);
    // the sketch: the m largest lane maxima (order keys, descending), from each
    // lane's rank among the 32 (ties by lane); tau, the mt-th largest, so that at
    // least mt tokens reach it and the unit's mt largest all do
    const uint32_t lkey = lm > -INFINITY ? f2key(lm) : 0u;
    uint32_t rank = 0;
#pragma unroll
    for (int o = 0; o < 32; ++o) {
        const uint32_t ok = __shfl_sync(0xffffffffu, lkey, o);
        rank += (ok > lkey || (ok == lkey && o < lane)) ? 1u : 0u;
    }
    const uint32_t nfin = __popc(__ballot_sync(0xffffffffu, lkey != 0u));
    const uint32_t m = min(uint32_t(ri.m), nfin);
    if (lkey != 0u && rank < m) {
        body->sketch[rank] = lkey;
        if (hist) atomicAdd(hist + key_bin(lkey), 1u);  // the row's histogram of sketch keys
    }
    // (a unit with fewer finite lane maxima than mt lists every finite token: only
    // then is its list sure to hold its top mt)
    const uint32_t at = __ballot_sync(0xffffffffu, nfin >= uint32_t(ri.mt) && rank == uint32_t(ri.mt) - 1u);
    uint32_t tau = at ? __shfl_sync(0xffffffffu, lkey, __ffs(at) - 1) : 0u;
    tau = max(tau, 1u);  // -inf (key 0 here) is never listed
    SLC_MARK(17);
    // list every finite token whose key reaches tau (x >= t as floats, -0 and
    // +0 alike, as the keys): one pass queues the vectors holding any (only
    // lanes whose maximum reaches tau can) with their bit masks, in order; the
    // list is then written from the queue, a vector per lane
    const float t = tau < 0x00800000u ? -FLT_MAX : key2f(tau);  // x >= t: finite and key >= tau
    const typename Vec<InT>::Thr t2 = Vec<InT>::thr(t);
    uint32_t total = 0;
    int nq = 0;
    // only the vectors of the lanes whose maximum reaches tau can hold such tokens
    // (vector j is lane j % 32's): they are spread over all 32 lanes, work item
    // w = i * na + a standing for vector i * 32 + (the a-th such lane)
    const uint32_t act = __ballot_sync(0xffffffffu, lkey >= tau);
    const int na = __popc(act);
    const int work = na * ((sv.nvec + 31) >> 5);
    const float inv_na = na ? 1.0f / float(na) : 0.0f;
#pragma unroll 1
    for (int w0 = 0; w0 < work; w0 += 32) {
        const int w = w0 + lane;
        const int i = int((float(w) + 0.5f) * inv_na);  // w / na, exact for these sizes
        const int j = i * 32 + nth_set_lane(act, w - i * na);
        const uint32_t hit = (w < work && j < sv.nvec) ? Vec<InT>::mask_ge(sv.vec(j), t2) : 0u;
        const uint32_t bal = __ballot_sync(0xffffffffu, hit != 0u);
        const int at = nq + __popc(bal & ((1u << lane) - 1u));
        if (hit && at < kTQCap) q[at] = (uint32_t(j) << 8) | hit;
        nq += __popc(bal);
        total += uint32_t(__popc(hit));
    }
    total = __reduce_add_sync(0xffffffffu, total);
    SLC_MARK(18);
    uint32_t xcount = 0;  // biased tokens that reach tau, listed after the others
    for (int q0 = 0; q0 < nx; q0 += 32) {
        const bool in = q0 + lane < nx && xv[q0 + lane] >= t;
        xcount += __popc(__ballot_sync(0xffffffffu, in));
    }
    const uint32_t total_nx = total;
    total += xcount;
    if (total <= uint32_t(kLCap)) {  // else the list is not kept (overflow)
        __syncwarp();
        uint32_t xbase = total_nx;
        for (int q0 = 0; q0 < nx; q0 += 32) {
            const bool in = q0 + lane < nx && xv[q0 + lane] >= t;
            const uint32_t bal = __ballot_sync(0xffffffffu, in);
            if (in) body->list[xbase + __popc(bal & ((1u << lane) - 1u))] = cand_word(f2key(xv[q0 + lane]), xi[q0 + lane]);
            xbase += __popc(bal);
        }
        uint32_t base = 0;
#pragma unroll 1
        for (int i0 = 0; i0 < nq; i0 += 32) {
            const int i = i0 + lane;
            const uint32_t w = i < nq ? q[i] : 0u;
            const uint32_t c = __popc(w & 255u);
            uint32_t incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            uint32_t pos = base + incl - c;
            if (c) {
                const int j = int(w >> 8);
                const uint4 v = sv.vec(j);
#pragma unroll 1
                for (uint32_t hit = w & 255u; hit; hit &= hit - 1u) {
                    const int e = __ffs(hit) - 1;
                    body->list[pos++] = cand_word(f2key(Vec<InT>::get(v, e)), sv.c0 + j * E + e);
                }
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    SLC_MARK(19);
    // top-p rows without top-k: the unit's softmax mass at its maximum (at T);
    // logprob outputs over the whole row: the same at the outputs' temperature
    float zsum = 0.0f, zlow = 0.0f;
    const bool fin = mx > -INFINITY && mx < INFINITY;
    if (ri.need_z && fin) unit_mass<InT>(sv, mx, ri.s2, zsum, zlow, xv, nx);
    if (lane == 0)
        *reinterpret_cast<uint4*>(&body->tau) = make_uint4(tau, __float_as_uint(zsum), __float_as_uint(zlow), m);
    if (ri.need_zo) {
        float os = 0.0f, ol = 0.0f;
        if (ri.need_z && ri.s2o == ri.s2) {
            os = zsum;
            ol = zlow;
        } else if (fin) {
            unit_mass<InT>(sv, mx, ri.s2o, os, ol, xv, nx);
        }
        if (lane == 0) *reinterpret_cast<uint4*>(&body->zos) = make_uint4(__float_as_uint(os), __float_as_uint(ol), 0u, 0u);
    }
    hdr_out.mx = mx;
    hdr_out.amax = amax;
    hdr_out.flags = flags;
    hdr_out.n = total > uint32_t(kLCap) ? kOverflow : total;
}

// ---------------------------------------------------------------- finishing
// A row is finished once, by one warp, usually with none of this code in the
// SM's instruction cache: a cold instruction costs far more than a hot one, so
// the finishing code is kept short (loops rolled, helpers out of line).
__device__ __forceinline__ int32_t status_of(uint32_t fl)
{
    if (fl & kFlagNonFinite) return kRowNonFinite;
    if (!(fl & kFlagAnyFinite)) return kRowAllNegInf;
    if (fl & kFlagTimeout) return kRowTimeout;
    return kRowOk;
}

__device__ __forceinline__ void write_out(const KernelParams& kp, int r, int token, int32_t status)
{
    kp.out_tokens[r] = status ? -1 : token;
    if (kp.out_status) kp.out_status[r] = status;
}

__device__ __forceinline__ SliceHdr ld_hdr(const SliceHdr* p)
{
    const uint4 u = __ldcg(reinterpret_cast<const uint4*>(p));
    SliceHdr h;
    h.mx = __uint_as_float(u.x);
    h.amax = int32_t(u.y);
    h.flags = u.z;
    h.n = u.w;
    return h;
}

// Exact (double-precision) Gumbel score of token v of the row, its logit read
// again and its Philox word recomputed.
template <typename InT>
static __device__ __noinline__ double exact_score(const KernelParams& kp, RowInfo ri, uint32_t off_lo,
                                                  uint32_t off_hi, int v)
{
    const RowPhilox rp = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, off_lo, off_hi);
    const float x = biased_logit<InT>(kp, ri, v);
    return gumbel_score_f64(x, ri.T, philox_word(rp, v));
}

// The pick from the best two candidates (composite keys; b may be 0): by their
// fp32 scores when those are further apart than their error bound, else by the
// exact scores.
template <typename InT>
__device__ __forceinline__ int pick_of(const KernelParams& kp, const RowInfo& ri, uint32_t off_lo, uint32_t off_hi,
                                       const K2& t)
{
    const int ia = cand_idx(t.a);
    if (t.b == 0ull) return ia;
    const float sa = gkey_score(t.a), sb = gkey_score(t.b);
    if (sa - sb > settle_eps(sa, sb)) return ia;
    const int ib = cand_idx(t.b);
    const double da = exact_score<InT>(kp, ri, off_lo, off_hi, ia);
    const double db = exact_score<InT>(kp, ri, off_lo, off_hi, ib);
    return (da > db || (da == db && ia < ib)) ? ia : ib;
}

__device__ __forceinline__ void finish_greedy(const SliceParams& P, int r, int& tok, int32_t& st)
{
    const int lane = threadIdx.x & 31;
    const SliceHdr* hd = P.hdr + size_t(r) * P.G;
    float m = -INFINITY;
    int mi = INT_MAX;
    uint32_t fl = 0;
#pragma unroll 1
    for (int b = lane; b < P.G; b += 32) {
        const SliceHdr h = ld_hdr(hd + b);
        fl |= h.flags;
        if (h.mx > m || (h.mx == m && h.amax < mi)) {
            m = h.mx;
            mi = h.amax;
        }
    }
    fl = warp_or(fl);
    warp_max_idx(m, mi);
    st = status_of(fl);
    tok = st ? -1 : mi;
    if (lane == 0) write_out(P.k, r, mi, st);
}

template <typename InT>
__device__ __forceinline__ void finish_plain(const SliceParams& P, const RowInfo& ri, int r, uint32_t off_lo,
                                             uint32_t off_hi, int& tok, int32_t& st_out)
{
    const int lane = threadIdx.x & 31;
    const SliceHdr* hd = P.hdr + size_t(r) * P.G;
    const SliceBody* bd = P.body + size_t(r) * P.G;
    K2 t{0ull, 0ull};
    uint32_t fl = 0;
#pragma unroll 1
    for (int b = lane; b < P.G; b += 32) {
        fl |= __ldcg(&hd[b].flags);
        const uint4 g = __ldcg(reinterpret_cast<const uint4*>(&bd[b].ga));
        k2_insert(t, (static_cast<unsigned long long>(g.y) << 32) | g.x);
        k2_insert(t, (static_cast<unsigned long long>(g.w) << 32) | g.z);
    }
    fl = warp_or(fl);
    k2_warp_reduce(t);
    const int32_t st = status_of(fl);
    int token = -1;
    if (!st) token = pick_of<InT>(P.k, ri, off_lo, off_hi, t);
    if (lane == 0) write_out(P.k, r, token, st);
    tok = token;
    st_out = st;
}

// The largest 16-bit prefix P with at least k keys >= P << 16 (so P << 16 is at
// most the k-th largest key), found two bits at a time: count3(c1, c2, c3, n)
// adds to n[i] how many of the lane's keys reach c_i, and the warp sums them.
template <typename Count3>
__device__ __forceinline__ uint32_t kth_prefix(uint32_t k, Count3 count3)
{
    uint32_t p = 0;
#pragma unroll 1
    for (int sh = 14; sh >= 0; sh -= 2) {
        uint32_t n[3] = {0u, 0u, 0u};
        count3((p | (1u << sh)) << 16, (p | (2u << sh)) << 16, (p | (3u << sh)) << 16, n);
        const uint32_t n1 = __reduce_add_sync(0xffffffffu, n[0]);
        const uint32_t n2 = __reduce_add_sync(0xffffffffu, n[1]);
        const uint32_t n3 = __reduce_add_sync(0xffffffffu, n[2]);
        p |= (n3 >= k ? 3u : n2 >= k ? 2u : n1 >= k ? 1u : 0u) << sh;
    }
    return p << 16;
}

__device__ __forceinline__ void count3_key(uint32_t key, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t (&n)[3])
{
    n[0] += key >= c1 ? 1u : 0u;
    n[1] += key >= c2 ? 1u : 0u;
    n[2] += key >= c3 ? 1u : 0u;
}

// B for a top-k row: the 16-bit prefix of the k-th largest sketch key over the
// row (the row holds at least k). sk: kSketch words per slice, meta[b].w of
// them valid. Each lane keeps the 16-bit prefixes of its NS slices' keys two
// to a register (NS = the fewest that cover G slices, so that no lane counts
// empty slots) and counts them with paired 16-bit compares. The answer lies
// between the smallest and the largest valid prefix (at least k keys reach the
// smallest), so the search keeps lo (at least k keys reach it) and hi (fewer
// do) from those two and cuts the range in four each round: few rounds, since
// the keys of one row span a narrow range of prefixes.
template <int NS>
__device__ __forceinline__ uint32_t sketch_bound_n(const uint32_t* sk, const uint4* meta, int G, int k,
                                                   const uint32_t* hist)
{
    const int lane = threadIdx.x & 31;
    constexpr int kPairs = kSketch / 2;
    uint32_t pk[NS][kPairs];
    uint32_t pmin = 0xFFFFu, pmax = 0u;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int b = lane + 32 * i;
        uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
        uint32_t mb = 0;
        if (b < G) {
            lo = *reinterpret_cast<const uint4*>(sk + b * kSketch);
            hi = *reinterpret_cast<const uint4*>(sk + b * kSketch + 4);
            mb = meta[b].w;
        }
        const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int q = 0; q < kPairs; ++q) {
            const uint32_t a = uint32_t(2 * q) < mb ? w[2 * q] >> 16 : 0u;
            const uint32_t c = uint32_t(2 * q + 1) < mb ? w[2 * q + 1] >> 16 : 0u;
            pk[i][q] = a | (c << 16);
        }
        // the sketch is in descending order: its first key is the largest, its
        // last valid one the smallest
        if (mb) {
            pmax = max(pmax, w[0] >> 16);
            pmin = min(pmin, w[min(mb, uint32_t(kSketch)) - 1u] >> 16);
        }
    }
    uint32_t lo = __reduce_min_sync(0xffffffffu, pmin);
    uint32_t hi = __reduce_max_sync(0xffffffffu, pmax) + 1u;
    if (hist) {
        // the bin that holds the k-th largest key, from the top (lane l holds
        // bins 255 - 8 l down to 248 - 8 l); the answer lies within it
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = hist[kHistBins - 1 - 8 * lane - i];
            sum += c[i];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const uint32_t at = __ballot_sync(0xffffffffu, incl >= uint32_t(k));
        int bin = 0;
        if (at) {
            const int src = __ffs(at) - 1;
            uint32_t run = incl - sum;
            int mine = -1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // the lane's top bin first
                run += c[i];
                if (mine < 0 && run >= uint32_t(k)) mine = kHistBins - 1 - 8 * lane - i;
            }
            bin = __shfl_sync(0xffffffffu, mine, src);
            // bin 0 reaches down to -inf, bin 255 up to +inf
            if (bin > 0) lo = max(lo, bin_lo_prefix(bin));
            if (bin < kHistBins - 1) hi = min(hi, bin_hi_prefix(bin));
        }
    }
#pragma unroll 1
    while (hi - lo > 1u) {
        const uint32_t d = hi - lo - 1u;
        uint32_t t[3], n[3];
#pragma unroll
        for (int j = 0; j < 3; ++j) t[j] = lo + 1u + (d * uint32_t(j + 1)) / 4u;  // in (lo, hi)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            // both halves of the threshold hold the candidate prefix (>= 1, so
            // empty slots, prefix 0, never count)
            const uint32_t tt = t[j] * 0x00010001u;
            uint32_t a = 0;  // two 16-bit counts (at most NS * kSketch / 2 each)
#pragma unroll
            for (int i = 0; i < NS; ++i)
#pragma unroll
                for (int q = 0; q < kPairs; ++q) a += __vsetgeu2(pk[i][q], tt);
            n[j] = __reduce_add_sync(0xffffffffu, (a & 0xFFFFu) + (a >> 16));
        }
        // counts fall as the threshold rises
        if (n[2] >= uint32_t(k)) {
            lo = t[2];
        } else if (n[1] >= uint32_t(k)) {
            lo = t[1];
            hi = t[2];
        } else if (n[0] >= uint32_t(k)) {
            lo = t[0];
            hi = t[1];
        } else {
            hi = t[0];
        }
    }
    return lo << 16;
}

static __device__ SLC_FIN_INLINE uint32_t sketch_bound(const uint32_t* sk, const uint4* meta, int G, int k,
                                                      const uint32_t* hist = nullptr)
{
    if (G <= 32) return sketch_bound_n<1>(sk, meta, G, k, hist);
    if (G <= 64) return sketch_bound_n<2>(sk, meta, G, k, hist);
    if (G <= 96) return sketch_bound_n<3>(sk, meta, G, k, hist);
    return sketch_bound_n<kSPL>(sk, meta, G, k, hist);
}

// Keep, stably and at the front, the words whose key reaches lo; returns how
// many were kept.
static __device__ SLC_FIN_INLINE int compact_ge(unsigned long long* c, int n, uint32_t lo)
{
    const int lane = threadIdx.x & 31;
    int kept = 0;
#pragma unroll 1
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        const unsigned long long w = i < n ? c[i] : 0ull;
        const bool keep = i < n && cand_key(w) >= lo;
        const uint32_t bal = __ballot_sync(0xffffffffu, keep);
        __syncwarp();
        if (keep) c[kept + __popc(bal & ((1u << lane) - 1u))] = w;
        kept += __popc(bal);
        __syncwarp();
    }
    return kept;
}

// Keep (at the front, in their order) the candidates whose key's top 16 bits
// reach those of the k-th largest key: the k largest words and their ties in
// that 16-bit bin. Returns how many were kept.
static __device__ SLC_FIN_INLINE int select_top(unsigned long long* c, int n, int k)
{
    const int lane = threadIdx.x & 31;
    const uint32_t lo = kth_prefix(uint32_t(k), [&](uint32_t c1, uint32_t c2, uint32_t c3, uint32_t(&m)[3]) {
        uint32_t part[2][3] = {};
        int i = lane;
#pragma unroll 1
        for (; i + 32 < n; i += 64) {
            count3_key(cand_key(c[i]), c1, c2, c3, part[0]);
            count3_key(cand_key(c[i + 32]), c1, c2, c3, part[1]);
        }
        if (i < n) count3_key(cand_key(c[i]), c1, c2, c3, part[0]);
#pragma unroll
        for (int j = 0; j < 3; ++j) m[j] = part[0][j] + part[1][j];
    });
    return compact_ge(c, n, lo);
}

// The min-p threshold on the logit, m + T ln(min_p) in double precision,
// rounded up to fp32 (x >= result exactly when x >= the double threshold).
static __device__ __noinline__ float minp_threshold(float m, float T, float minp)
{
    const double th = double(m) + double(T) * log(double(minp));
    float t = float(th);
    if (double(t) < th) t = nextafterf(t, INFINITY);
    return t;
}

// ---- per-row logprob outputs
constexpr float kLn2 = 0.6931471805599453f;

// An error row: NaN logprobs, ids -1 (lane 0 and the first top_n lanes write).
__device__ __forceinline__ void lp_write_error(const KernelParams& kp, int r)
{
    const int lane = threadIdx.x & 31;
    if (lane == 0 && kp.out_tok_lp) kp.out_tok_lp[r] = __uint_as_float(0x7FC00000u);
    if (lane < kp.top_n) {
        kp.out_top_ids[size_t(r) * kp.top_n + lane] = -1;
        kp.out_top_lp[size_t(r) * kp.top_n + lane] = __uint_as_float(0x7FC00000u);
    }
}

// The outputs of row r from its sorted candidates (the first nc of `srt`, all
// of them carrying mass), its maximum m, log2 of its mass lz2 (both at the
// outputs' temperature, scale s2o) and the sampled token's logit xt.
__device__ __forceinline__ void lp_write(const KernelParams& kp, int r, const unsigned long long* srt, int nc,
                                         float m, float s2o, float lz2, float xt)
{
    const int lane = threadIdx.x & 31;
    if (lane == 0 && kp.out_tok_lp) kp.out_tok_lp[r] = ((xt - m) * s2o - lz2) * kLn2;
    if (lane < kp.top_n) {
        int id = -1;
        float lp = -INFINITY;
        if (lane < nc) {
            const unsigned long long c = srt[lane];
            id = cand_idx(c);
            lp = ((key2f(cand_key(c)) - m) * s2o - lz2) * kLn2;
        }
        kp.out_top_ids[size_t(r) * kp.top_n + lane] = id;
        kp.out_top_lp[size_t(r) * kp.top_n + lane] = lp;
    }
}

// Sort n words in warp-private shared memory, descending (bitonic through
// shared memory, padded with zeros up to a power of two; the buffer holds it).
static __device__ SLC_FIN_INLINE void warp_sort_smem(unsigned long long* a, int n)
{
    const int lane = threadIdx.x & 31;
    int np2 = 1;
    while (np2 < n) np2 <<= 1;
#pragma unroll 1
    for (int i = n + lane; i < np2; i += 32) a[i] = 0ull;
    __syncwarp();
#pragma unroll 1
    for (int size = 2; size <= np2; size <<= 1) {
#pragma unroll 1
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll 1
            for (int t = lane; t < (np2 >> 1); t += 32) {
                const int lo = ((t & ~(stride - 1)) << 1) | (t & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long x = a[lo], y = a[hi];
                if ((x < y) == desc) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncwarp();
        }
    }
}

// The first `keep` of n distinct words in descending order, out[rank] = word:
// each word's rank is the number of larger words, counted by its lane against
// every word (broadcast reads, four partial counts).
static __device__ SLC_FIN_INLINE void rank_sort(const unsigned long long* c, int n, unsigned long long* out, int keep)
{
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        const unsigned long long w = i < n ? c[i] : ~0ull;
        int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        int j = 0;
#pragma unroll 1
        for (; j + 4 <= n; j += 4) {
            r0 += c[j] > w ? 1 : 0;
            r1 += c[j + 1] > w ? 1 : 0;
            r2 += c[j + 2] > w ? 1 : 0;
            r3 += c[j + 3] > w ? 1 : 0;
        }
#pragma unroll 1
        for (; j < n; ++j) r0 += c[j] > w ? 1 : 0;
        const int rank = r0 + r1 + r2 + r3;
        if (i < n && rank < keep) out[rank] = w;
    }
    __syncwarp();
}

// Inclusive warp scan of a 64-bit count.
__device__ __forceinline__ unsigned long long warp_incl_u64(unsigned long long v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    return v;
}

// The cuts over the sorted candidates of a truncated row, each keeping a prefix
// (top-k, then top-p over the top-k set or the whole row, then min-p), and the
// Gumbel pick over what is kept. Returns false when top-p reaches past the
// candidates of a row without top-k or min-p (the exact path takes it).
// hs / meta: the slices' staged headers and (tau, zs, zc, m) words.
template <typename InT>
static __device__ SLC_FIN_INLINE bool cut_and_pick(const SliceParams& P, const RowInfo& ri, int r, uint32_t off_lo,
                                                 uint32_t off_hi, const unsigned long long* cand, int C, float m,
                                                 float xthr, const SliceHdr* hs, const uint4* meta, int& tok_out)
{
    const int lane = threadIdx.x & 31;
    const int nk = ri.do_topk ? ri.k : C;
    int nkeep = nk;
    if (ri.do_topp) {
        // fixed-point masses (2^-40 units of exp((x - m) / T)); keep while the
        // exclusive prefix mass is below p * Z, i.e. below tq = ceil(p * Zq)
        double Zq;
        if (ri.do_topk) {
            unsigned long long s = 0;
#pragma unroll 1
            for (int i = lane; i < nk; i += 32) s += mass_q(key2f(cand_key(cand[i])), m, ri.invT);
            Zq = double(warp_sum_u64(s));
        } else {
            double z = 0.0;
#pragma unroll 1
            for (int b = lane; b < P.G; b += 32) {
                const float mx = hs[b].mx;
                if (mx > -INFINITY)
                    z += (double(__uint_as_float(meta[b].y)) + double(__uint_as_float(meta[b].z))) *
                         double(exp2f((mx - m) * ri.s2));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
            Zq = z * 0x1p40;
        }
        const unsigned long long tq = __double2ull_ru(double(ri.p) * Zq);
        unsigned long long base = 0;
        int cut = nk;
#pragma unroll 1
        for (int i0 = 0; i0 < nk; i0 += 32) {
            const int i = i0 + lane;
            const unsigned long long q = i < nk ? mass_q(key2f(cand_key(cand[i])), m, ri.invT) : 0ull;
            const unsigned long long incl = warp_incl_u64(q);
            const unsigned long long excl = base + incl - q;
            const uint32_t sb = __ballot_sync(0xffffffffu, i < nk && i > 0 && !(excl < tq));
            if (sb) {
                cut = i0 + __ffs(sb) - 1;
                break;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (!ri.do_topk && !ri.do_minp && cut == nk) return false;  // the cut lies past the candidates
        nkeep = cut;
    }
    if (ri.do_minp) {
        int c = 0;
#pragma unroll 1
        for (int i = lane; i < nkeep; i += 32) c += key2f(cand_key(cand[i])) >= xthr ? 1 : 0;
        nkeep = min(nkeep, int(__reduce_add_sync(0xffffffffu, uint32_t(c))));
    }
    nkeep = max(nkeep, 1);
    SLC_MARK(14);
    int token;
    if (ri.greedy) {
        token = cand_idx(cand[0]);  // a greedy row here only for its logprob outputs
    } else {
        // Gumbel-max over the kept prefix
        const RowPhilox rp = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, off_lo, off_hi);
        K2 t{0ull, 0ull};
#pragma unroll 1
        for (int i = lane; i < nkeep; i += 32) {
            const unsigned long long c = cand[i];
            const int v = cand_idx(c);
            k2_insert(t, gkey(score2(key2f(cand_key(c)), ri.s2, philox_word(rp, v)), v));
        }
        k2_warp_reduce(t);
        token = pick_of<InT>(P.k, ri, off_lo, off_hi, t);
    }
    if (lane == 0) write_out(P.k, r, token, kRowOk);
    tok_out = token;
    if (row_lp(ri) && !P.k.lp_unscaled) {
        // the kept set's mass at the outputs' temperature, and the token's logit
        double z = 0.0;
        float xt = 0.0f;
#pragma unroll 1
        for (int i = lane; i < nkeep; i += 32) {
            const unsigned long long c = cand[i];
            const float x = key2f(cand_key(c));
            z += double(exp2f((x - m) * ri.s2o));
            if (cand_idx(c) == token) xt = x;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            z += __shfl_xor_sync(0xffffffffu, z, off);
            xt += __shfl_xor_sync(0xffffffffu, xt, off);
        }
        lp_write(P.k, r, cand, min(nkeep, P.k.top_n), m, ri.s2o, log2f(float(z)), xt);
    }
    return true;
}

__device__ __forceinline__ void cp_async_commit_wait()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gsrc)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}

// Vector j of a slice that is not 16-byte aligned, or the ragged last one, read
// element by element (-inf past the slice).
template <typename InT>
static __device__ __noinline__ uint4 load_vec_slow(const InT* g, int j, int n)
{
    SliceView<InT> sv;
    sv.sm = nullptr;
    sv.g = g;
    sv.nb = 0;
    sv.nvec = 0;
    sv.n = n;
    sv.c0 = 0;
    return sv.vec(j);
}

// Append to the candidates c[C0..) the finite tokens >= B (order key) of the
// nre slices listed in re[], reading them again from global memory: 8 vectors
// per lane in flight, counted, then written at their warp-wide positions.
// Returns the new count (more than cap when they do not fit).
template <typename InT>
static __device__ __noinline__ int reread_slices(const SliceParams& P, RowInfo ri, const uint16_t* re,
                                                 int nre, uint32_t B, unsigned long long* c, int C0, int cap,
                                                 int32_t* xi, float* xv)
{
    constexpr int E = Vec<InT>::E;
    constexpr int U = 8;
    const int lane = threadIdx.x & 31;
    const int V = int(P.k.vocab);
    const int nvW = (P.W + E - 1) / E;
    const int total = nre * nvW;
    // x >= tB exactly when x is not -inf and its key reaches B
    const float tB = B < 0x00800000u ? -FLT_MAX : key2f(B);
    const typename Vec<InT>::Thr t2 = Vec<InT>::thr(tB);
    // logit_bias / min_tokens: the row's biased and banned tokens are taken
    // apart (their raw logits skipped below, their values appended at the end)
    const int nx = has_extras(P.k) ? max(0, row_extras<InT>(P.k, ri, 0, V, xi, xv)) : 0;
    int C = C0;
#pragma unroll 1
    for (int base = 0; base < total; base += 32 * U) {
        uint4 v[U];
        int t0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int f = base + u * 32 + lane;
            const int si = f / nvW;
            const int j = f - si * nvW;
            const int b = f < total ? int(re[si]) : 0;
            const int c0 = b * P.W;
            const int n = min(P.W, V - c0);
            const InT* g = slice_ptr<InT>(P.k, ri.lrow, c0);
            t0[u] = c0 + j * E;
            v[u] = Vec<InT>::neg_inf();
            if (f < total && j * E < n) {
                if ((reinterpret_cast<uintptr_t>(g) & 15u) == 0 && (j + 1) * E <= n)
                    v[u] = __ldg(reinterpret_cast<const uint4*>(g) + j);
                else
                    v[u] = load_vec_slow<InT>(g, j, n);
                if (sanitizing(P.k)) v[u] = Vec<InT>::sanitized(v[u]);
                if (mask_of(P.k)) {
                    const int tk = c0 + j * E;
                    const uint32_t w = __ldg(mask_of(P.k) + size_t(ri.r) * size_t(P.k.mask_stride) + (tk >> 5));
                    v[u] = Vec<InT>::masked(v[u], (w >> (tk & 31)) & ((1u << E) - 1u));
                }
            }
        }
        uint32_t hits[U];
        uint32_t mine = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t h = Vec<InT>::mask_ge(v[u], t2);
            if (nx)
                for (uint32_t b2 = h; b2; b2 &= b2 - 1u) {
                    const int e = __ffs(b2) - 1;
                    if (is_extra(xi, nx, t0[u] + e)) h &= ~(1u << e);
                }
            hits[u] = h;
            mine += __popc(h);
        }
        SLC_MARK(15);
        uint32_t incl = mine;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        uint32_t pos = uint32_t(C) + incl - mine;
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll 1
            for (uint32_t hit = hits[u]; hit; hit &= hit - 1u) {
                const int e = __ffs(hit) - 1;
                if (pos < uint32_t(cap)) c[pos] = cand_word(f2key(Vec<InT>::get(v[u], e)), t0[u] + e);
                ++pos;
            }
        }
        C += int(__shfl_sync(0xffffffffu, incl, 31));
    }
    // the biased tokens of the slices read again that reach B
    for (int q0 = 0; q0 < nx; q0 += 32) {
        const int q = q0 + lane;
        bool in = false;
        if (q < nx && xv[q] >= tB) {
            const int b = xi[q] / P.W;
            for (int i = 0; i < nre; ++i) in |= int(re[i]) == b;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, in);
        const uint32_t pos = uint32_t(C) + __popc(bal & ((1u << lane) - 1u));
        if (in && pos < uint32_t(cap)) c[pos] = cand_word(f2key(xv[q]), xi[q]);
        C += __popc(bal);
    }
    __syncwarp();
    return C;
}

// A truncated row from its slices' records. The warp's staging slot (idle at
// this point) is its scratch: the slices' headers, (tau, zs, zc, m) words and
// sketches in one round of copies; then, over the sketches, the lists of the
// slices that matter in a second round, which become the candidates. Returns
// false when the row must take the exact path (m out).
template <typename InT>
static __device__ SLC_FIN_INLINE bool finish_trunc(const SliceParams& P, WarpScratch& ws, const RowInfo& ri, int r,
                                                 uint32_t off_lo, uint32_t off_hi, unsigned char* scratch,
                                                 float& m_out, int& tok, int32_t& st_out)
{
    const int lane = threadIdx.x & 31;
    const int G = P.G;
    const SliceHdr* hd = P.hdr + size_t(r) * G;
    const SliceBody* bd = P.body + size_t(r) * G;
    SliceHdr* hs = reinterpret_cast<SliceHdr*>(scratch);            // [G]
    uint4* meta = reinterpret_cast<uint4*>(scratch + size_t(G) * 16);  // [G]
    uint32_t* sk = reinterpret_cast<uint32_t*>(scratch + size_t(G) * 32);  // [G][kSketch]
    unsigned long long* area = reinterpret_cast<unsigned long long*>(sk);  // the lists, over the sketches
    const int cap = int((size_t(kSlotBytes) - size_t(32) * G) / 8);
    // the row's histogram of sketch keys, at the end of the slot (read before the
    // lists reach it)
    uint32_t* hist = P.cnt + size_t(r) * kCntStride + kHistOff;
    uint32_t* hsm = reinterpret_cast<uint32_t*>(scratch + kSlotBytes - kHistBins * 4);
    // round 1
    cp_async16(hsm + 8 * lane, hist + 8 * lane);
    cp_async16(hsm + 8 * lane + 4, hist + 8 * lane + 4);
#pragma unroll 1
    for (int b = lane; b < G; b += 32) {
        cp_async16(hs + b, hd + b);
        cp_async16(meta + b, &bd[b].tau);
        cp_async16(sk + b * kSketch, &bd[b].sketch[0]);
        cp_async16(sk + b * kSketch + 4, &bd[b].sketch[4]);
    }
    cp_async_commit_wait();
    // the histogram is zero again for the next launch
    reinterpret_cast<uint4*>(hist)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(hist)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    SLC_MARK(7);
    uint32_t fl = 0, nkeys = 0, taumax = 0;
    float m = -INFINITY;
    int mi = INT_MAX;
#pragma unroll 1
    for (int b = lane; b < G; b += 32) {
        const SliceHdr h = hs[b];
        fl |= h.flags;
        nkeys += meta[b].w;
        taumax = max(taumax, meta[b].x);
        if (h.mx > m || (h.mx == m && h.amax < mi)) {
            m = h.mx;
            mi = h.amax;
        }
    }
    fl = warp_or(fl);
    nkeys = __reduce_add_sync(0xffffffffu, nkeys);
    taumax = __reduce_max_sync(0xffffffffu, taumax);
    warp_max_idx(m, mi);
    m_out = m;
    const int32_t st = status_of(fl);
    st_out = st;
    tok = -1;
    if (st) {
        if (lane == 0) write_out(P.k, r, -1, st);
        if (row_lp(ri)) lp_write_error(P.k, r);
        return true;
    }
    // the min-p threshold on the logit: m + T ln(min_p), rounded up to fp32
    float xthr = -INFINITY;
    if (ri.do_minp) xthr = minp_threshold(m, ri.T, ri.minp);
    // B: every kept token's key reaches it
    uint32_t B;
    if (ri.do_topk) {
        if (ri.k > kKCap || nkeys < uint32_t(ri.k)) return false;
        B = sketch_bound(sk, meta, G, ri.k, hsm);
    } else if (ri.do_minp) {
        B = f2key(xthr);
    } else {
        B = taumax;
    }
    B = max(B, 1u);
    SLC_MARK(8);
    __syncwarp();
    // round 2: the lists of the slices that reach B and are complete above it
    // (or, on a top-k row with k <= kKComplete, complete for the row's top k),
    // side by side; the others are read again below
    const bool topk_complete = ri.do_topk && ri.k <= kKComplete;
    uint32_t total = 0, nre = 0;
#pragma unroll 1
    for (int c0 = 0; c0 < G; c0 += 32) {
        const int b = c0 + lane;
        uint32_t n = 0;
        bool again = false;
        if (b < G) {
            const SliceHdr h = hs[b];
            if (h.mx > -INFINITY && f2key(h.mx) >= B) {
                if (h.n == kOverflow || (meta[b].x > B && !topk_complete)) again = true;
                else n = h.n;
            }
        }
        uint32_t incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const uint32_t pos = total + incl - n;
        if (pos + n <= uint32_t(cap)) {
#pragma unroll 1
            for (uint32_t e = 0; e < n; ++e) cp_async8(area + pos + e, &bd[b].list[e]);
        }
        const uint32_t who = __ballot_sync(0xffffffffu, again);
        const uint32_t at = nre + __popc(who & ((1u << lane) - 1u));
        if (again && at < uint32_t(kReCap)) ws.re[at] = uint16_t(b);
        nre += __popc(who);
        total += __shfl_sync(0xffffffffu, incl, 31);
    }
    cp_async_commit_wait();
    __syncwarp();
    if (total > uint32_t(cap) || nre > uint32_t(kReCap)) return false;
    int C = compact_ge(area, int(total), B);
    SLC_MARK(9);
    if (nre) C = reread_slices<InT>(P, ri, ws.re, int(nre), B, area, C, cap, ws.xi, ws.xv);
    SLC_MARK(10);
    if (C > cap) return false;
    if (ri.do_topk && C < ri.k) return false;
    const unsigned long long* sorted = area;
    if (C <= kRankSortMax && 2 * C <= cap) {
        // sorted copy after the candidates; a top-k row keeps only its k largest
        const int keep = ri.do_topk ? ri.k : C;
        rank_sort(area, C, area + C, keep);
        sorted = area + C;
        C = keep;
    } else {
        // top-k: bring the k largest to the front first
        if (ri.do_topk && C > ri.k) C = select_top(area, C, ri.k);
        int np2 = 1;
        while (np2 < C) np2 <<= 1;
        if (np2 > cap) return false;
        warp_sort_smem(area, C);
    }
    SLC_MARK(11);
    return cut_and_pick<InT>(P, ri, r, off_lo, off_hi, sorted, C, m, xthr, hs, meta, tok);
}

// The logprob outputs of row r over its whole vocabulary at the outputs'
// temperature (untruncated rows, and every row when they are unscaled): the mass
// from the units' records, the top n from their lists (each unit lists at least
// its top n, so a list that did not overflow holds every token of the row's top
// n in its slice). `token` is the sampled one; st its status.
template <typename InT>
static __device__ __noinline__ bool finish_lp_row(const SliceParams& P, WarpScratch& ws, RowInfo ri, int r,
                                                  int token, int32_t st, unsigned char* scratch, float& m_out)
{
    const int lane = threadIdx.x & 31;
    const KernelParams& kp = P.k;
    if (st) {
        lp_write_error(kp, r);
        return true;
    }
    const int G = P.G;
    const int n = kp.top_n;
    const SliceHdr* hd = P.hdr + size_t(r) * G;
    const SliceBody* bd = P.body + size_t(r) * G;
    SliceHdr* hs = reinterpret_cast<SliceHdr*>(scratch);                   // [G]
    uint4* meta = reinterpret_cast<uint4*>(scratch + size_t(G) * 16);        // [G] (tau, zs, zc, m)
    uint4* zo = reinterpret_cast<uint4*>(scratch + size_t(G) * 32);          // [G] (zos, zoc, -, -)
    uint32_t* sk = reinterpret_cast<uint32_t*>(scratch + size_t(G) * 48);    // [G][kSketch]
    unsigned long long* area = reinterpret_cast<unsigned long long*>(sk);  // the lists, over the sketches
    const int cap = int((size_t(kSlotBytes) - size_t(48) * G) / 8);
#pragma unroll 1
    for (int b = lane; b < G; b += 32) {
        cp_async16(hs + b, hd + b);
        cp_async16(meta + b, &bd[b].tau);
        cp_async16(zo + b, &bd[b].zos);
        cp_async16(sk + b * kSketch, &bd[b].sketch[0]);
        cp_async16(sk + b * kSketch + 4, &bd[b].sketch[4]);
    }
    cp_async_commit_wait();
    __syncwarp();
    float m = -INFINITY;
    uint32_t nkeys = 0;
#pragma unroll 1
    for (int b = lane; b < G; b += 32) {
        m = fmaxf(m, hs[b].mx);
        nkeys += meta[b].w;
    }
    m = __shfl_sync(0xffffffffu, key2f(__reduce_max_sync(0xffffffffu, f2key(m))), 0);
    m_out = m;
    nkeys = __reduce_add_sync(0xffffffffu, nkeys);
    double z = 0.0;
#pragma unroll 1
    for (int b = lane; b < G; b += 32) {
        const float mx = hs[b].mx;
        if (mx > -INFINITY)
            z += (double(__uint_as_float(zo[b].x)) + double(__uint_as_float(zo[b].y))) *
                 double(exp2f((mx - m) * ri.s2o));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    const float lz2 = log2f(float(z));
    const float xt = biased_logit<InT>(kp, ri, token);
    int C = 0;
    if (n > 0) {
        // B: the 16-bit prefix of the n-th largest sketch key (all listed tokens
        // when the sketches hold fewer)
        uint32_t B = nkeys >= uint32_t(n) ? sketch_bound(sk, meta, G, n) : 1u;
        B = max(B, 1u);
        __syncwarp();
        uint32_t total = 0, nre = 0;
#pragma unroll 1
        for (int c0 = 0; c0 < G; c0 += 32) {
            const int b = c0 + lane;
            uint32_t cnt = 0;
            bool again = false;
            if (b < G) {
                const SliceHdr h = hs[b];
                if (h.mx > -INFINITY && f2key(h.mx) >= B) {
                    if (h.n == kOverflow) again = true;
                    else cnt = h.n;
                }
            }
            uint32_t incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            const uint32_t pos = total + incl - cnt;
            if (pos + cnt <= uint32_t(cap)) {
#pragma unroll 1
                for (uint32_t e = 0; e < cnt; ++e) cp_async8(area + pos + e, &bd[b].list[e]);
            }
            const uint32_t who = __ballot_sync(0xffffffffu, again);
            const uint32_t at = nre + __popc(who & ((1u << lane) - 1u));
            if (again && at < uint32_t(kReCap)) ws.re[at] = uint16_t(b);
            nre += __popc(who);
            total += __shfl_sync(0xffffffffu, incl, 31);
        }
        cp_async_commit_wait();
        __syncwarp();
        bool ok = total <= uint32_t(cap) && nre <= uint32_t(kReCap);
        if (ok) {
            C = compact_ge(area, int(total), B);
            if (nre) C = reread_slices<InT>(P, ri, ws.re, int(nre), B, area, C, cap, ws.xi, ws.xv);
            ok = C <= cap && 2 * C <= cap && C <= kRankSortMax;
        }
        if (!ok) return false;  // more candidates than the lists settle here (ties): the exact path
        rank_sort(area, C, area + C, min(C, n));
        area += C;
        C = min(C, n);
    }
    lp_write(kp, r, area, C, m, ri.s2o, lz2, xt);
    return true;
}

// ---------------------------------------------------------------- exact path (whole CTA)
__device__ __forceinline__ unsigned long long cta_suffix_scan(unsigned long long v, SliceShared& sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long s = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_down_sync(0xffffffffu, s, off);
        if (lane + off < 32) s += o;
    }
    if (lane == 0) sh.scan_w[wid] = s;
    __syncthreads();
    unsigned long long later = 0;
    for (int w = wid + 1; w < kW; ++w) later += sh.scan_w[w];
    __syncthreads();
    return s + later;
}

__device__ __forceinline__ int cta_excl_scan(int v, int& total, SliceShared& sh)
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
    for (int w = 0; w < kW; ++w) {
        if (w < wid) before += sh.red_i[w];
        tot += sh.red_i[w];
    }
    __syncthreads();
    total = tot;
    return before + s - v;
}

// Token v of the row: sanitised, masked, and taken from the CTA's table (set
// up by cta_bias_setup) when the row carries logit_bias or a min_tokens ban.
template <typename InT>
__device__ __forceinline__ float row_x(const KernelParams& kp, const RowInfo& ri, int v, const SliceShared& sh)
{
    float x = ElemTraits<InT>::load(kp.logits, int64_t(ri.lrow) * kp.row_stride + v);
    if (sanitizing(kp) && x != x) x = -INFINITY;
    if (mask_of(kp) && !((__ldg(mask_of(kp) + size_t(ri.r) * size_t(kp.mask_stride) + (v >> 5)) >> (v & 31)) & 1u))
        return -INFINITY;
    if (sh.bx_n && ((sh.bx_bits[v >> 5] >> (v & 31)) & 1u))
        for (int q = 0; q < sh.bx_n; ++q)
            if (sh.bx_i[q] == v) return sh.bx_v[q];
    return x;
}

// The row's logit_bias and min_tokens ban for the CTA's exact path: its biased
// and banned tokens (warp 0) and their bitmap in the idle staging slots.
template <typename InT>
__device__ __forceinline__ void cta_bias_setup(SliceShared& sh, unsigned char* slots, const KernelParams& kp,
                                               const RowInfo& ri)
{
    const int tid = threadIdx.x, V = int(kp.vocab);
    if (!has_extras(kp)) {
        if (tid == 0) sh.bx_n = 0;
        __syncthreads();
        return;
    }
    uint32_t* bits = reinterpret_cast<uint32_t*>(slots);
    for (int w = tid; w < (V + 31) / 32; w += kT) bits[w] = 0u;
    if (tid < 32) {
        const int n = max(0, row_extras<InT>(kp, ri, 0, V, sh.bx_i, sh.bx_v));
        if (tid == 0) {
            sh.bx_n = n;
            sh.bx_bits = bits;
        }
    }
    __syncthreads();
    for (int q = tid; q < sh.bx_n; q += kT) atomicOr(&bits[sh.bx_i[q] >> 5], 1u << (sh.bx_i[q] & 31));
    __syncthreads();
}

// The token closing the kept prefix: the first token (value desc, index asc)
// whose inclusive weight (count, or fixed-point mass) reaches the target.
// Tokens outside the domain prefix (dkey, didx) weigh nothing when dom is set.
template <typename InT>
__device__ void cta_select(SliceShared& sh, const KernelParams& kp, const RowInfo& ri, int V, bool mass_mode,
                           bool dom, uint32_t dkey, int didx, float m, unsigned long long count_target,
                           uint32_t& out_key, int& out_idx)
{
    const int tid = threadIdx.x;
    if (tid == 0) {
        sh.sel_prefix = 0;
        sh.sel_wabove = 0;
        sh.sel_target = count_target;
    }
    __syncthreads();
    uint32_t pbits = 0;
    for (int level = 0; level < 4; ++level) {
        for (int i = tid; i < 256; i += kT) {
            sh.hcnt[i] = 0;
            sh.hmass[i] = 0;
        }
        __syncthreads();
        const uint32_t prefix = uint32_t(sh.sel_prefix);
        const int shift = 24 - 8 * level;
        for (int v = tid; v < V; v += kT) {
            const float x = row_x<InT>(kp, ri, v, sh);
            if (!(x > -INFINITY)) continue;
            const uint32_t key = f2key(x);
            if (dom && !in_prefix(key, v, dkey, didx)) continue;
            if (pbits && (key >> (32 - pbits)) != prefix) continue;
            const uint32_t d = (key >> shift) & 255u;
            atomicAdd(&sh.hcnt[d], 1u);
            if (mass_mode) atomicAdd(&sh.hmass[d], mass_q(x, m, ri.invT));
        }
        __syncthreads();
        const int d = tid < 256 ? tid : 0;
        const unsigned long long wgt = tid < 256 ? (mass_mode ? sh.hmass[d] : (unsigned long long)sh.hcnt[d]) : 0ull;
        const unsigned long long incl = cta_suffix_scan(wgt, sh);
        if (tid == 0 && mass_mode && level == 0) {
            unsigned long long t = (unsigned long long)ceil(double(ri.p) * double(incl));
            sh.sel_target = t < 1 ? 1 : t;
        }
        __syncthreads();
        const unsigned long long target = sh.sel_target, wa = sh.sel_wabove;
        __syncthreads();
        if (tid < 256 && wgt > 0 && wa + incl >= target && wa + (incl - wgt) < target) {
            sh.sel_prefix = (unsigned long long)((prefix << 8) | uint32_t(d));
            sh.sel_wabove = wa + (incl - wgt);
        }
        __syncthreads();
        pbits += 8;
    }
    const uint32_t K = uint32_t(sh.sel_prefix);
    unsigned long long tie_J;
    {
        const unsigned long long wt = mass_mode ? mass_q(key2f(K), m, ri.invT) : 1ull;
        tie_J = (sh.sel_target - sh.sel_wabove + wt - 1) / wt;
    }
    // the tie_J-th token (index order) holding key K
    int base = 0;
    for (int v0 = 0; v0 < V; v0 += kT) {
        const int v = v0 + tid;
        int c = 0;
        if (v < V) {
            const float x = row_x<InT>(kp, ri, v, sh);
            const uint32_t key = f2key(x);
            c = (x > -INFINITY && key == K && (!dom || in_prefix(key, v, dkey, didx))) ? 1 : 0;
        }
        int total = 0;
        const int excl = cta_excl_scan(c, total, sh);
        if (c && (unsigned long long)(base + excl + 1) == tie_J) sh.sel_idx = v;
        base += total;
        if ((unsigned long long)base >= tie_J) break;
    }
    __syncthreads();
    out_key = K;
    out_idx = sh.sel_idx;
    __syncthreads();
}

template <typename InT>
__device__ __noinline__ void cta_exact_row(SliceShared& sh, unsigned char* slots, const SliceParams& P, int r,
                                           RowInfo ri, float m, uint32_t off_lo, uint32_t off_hi)
{
    const KernelParams& kp = P.k;
    const int V = int(kp.vocab);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    cta_bias_setup<InT>(sh, slots, kp, ri);
    uint32_t bk = 0;
    int bi = 0;
    bool hb = false;
    if (ri.do_topk) {
        cta_select<InT>(sh, kp, ri, V, false, false, 0u, 0, m, (unsigned long long)ri.k, bk, bi);
        hb = true;
    }
    if (ri.do_topp) {
        cta_select<InT>(sh, kp, ri, V, true, hb, bk, bi, m, 0ull, bk, bi);
        hb = true;
    }
    float xthr = -INFINITY;
    if (ri.do_minp) {
        const double th = double(m) + double(ri.T) * log(double(ri.minp));
        float f = float(th);
        if (double(f) < th) f = nextafterf(f, INFINITY);
        xthr = f;
    }
    // the pick (greedy rows: the maximum, lowest index) and the kept set's mass
    // and size at the outputs' temperature (logprob outputs over the kept set)
    const bool lp_kept = row_lp(ri) && !kp.lp_unscaled && ri.cls == kClsTrunc;
    const RowPhilox rp = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, off_lo, off_hi);
    K2 t{0ull, 0ull};
    double z = 0.0;
    uint32_t nk = 0;
    for (int v = tid; v < V; v += kT) {
        const float x = row_x<InT>(kp, ri, v, sh);
        if (!(x > -INFINITY)) continue;
        const bool kept = !(hb && !in_prefix(f2key(x), v, bk, bi)) && !(ri.do_minp && !(x >= xthr));
        if (row_lp(ri) && (kept || !lp_kept)) {
            z += double(exp2f((x - m) * ri.s2o));
            ++nk;
        }
        if (!kept) continue;
        if (ri.greedy) k2_insert(t, cand_word(f2key(x), v));
        else k2_insert(t, gkey(score2(x, ri.s2, philox_word(rp, v)), v));
    }
    k2_warp_reduce(t);
    if (lane == 0) {
        sh.red_k[2 * wid] = t.a;
        sh.red_k[2 * wid + 1] = t.b;
    }
    if (row_lp(ri)) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        nk = __reduce_add_sync(0xffffffffu, nk);
        if (lane == 0) {
            sh.red_d[wid] = z;
            sh.red_i[wid] = int(nk);
        }
    }
    __syncthreads();
    if (wid == 0) {
        K2 a{0ull, 0ull};
        if (lane < kW) {
            a.a = sh.red_k[2 * lane];
            a.b = sh.red_k[2 * lane + 1];
        }
        k2_warp_reduce(a);
        const int token = ri.greedy ? cand_idx(a.a) : pick_of<InT>(kp, ri, off_lo, off_hi, a);
        if (lane == 0) {
            write_out(kp, r, token, kRowOk);
            if (P.stats) atomicAdd(P.stats, 1ull);
            sh.sel_idx = token;
        }
    }
    __syncthreads();
    if (!row_lp(ri)) return;
    // logprob outputs: the first n of the kept set (or of the row) in (value desc,
    // index asc) order, from the n-th of that order; the kept set is a prefix of it
    double zt = 0.0;
    int nkt = 0;
    for (int w = 0; w < kW; ++w) {
        zt += sh.red_d[w];
        nkt += sh.red_i[w];
    }
    const int token = sh.sel_idx;
    const int n = min(kp.top_n, nkt);
    __syncthreads();
    if (tid == 0) sh.lp_cnt = 0;
    uint32_t nkey = 0;
    int nidx = 0;
    if (n > 0) cta_select<InT>(sh, kp, ri, V, false, false, 0u, 0, m, (unsigned long long)n, nkey, nidx);
    __syncthreads();
    if (n > 0) {
        for (int v = tid; v < V; v += kT) {
            const float x = row_x<InT>(kp, ri, v, sh);
            if (x > -INFINITY && in_prefix(f2key(x), v, nkey, nidx)) {
                const int q = atomicAdd(&sh.lp_cnt, 1);
                if (q < kMaxTopN) sh.lp_list[q] = cand_word(f2key(x), v);
            }
        }
    }
    __syncthreads();
    if (wid == 0) {
        // rank the (at most n) collected words: word `lane` goes to its rank
        const int c = min(sh.lp_cnt, n);
        unsigned long long w = 0ull;
        int rank = 0;
        if (lane < c) {
            w = sh.lp_list[lane];
            for (int j = 0; j < c; ++j) rank += sh.lp_list[j] > w ? 1 : 0;
        }
        __syncwarp();
        if (lane < c) sh.lp_list[rank] = w;
        __syncwarp();
        const float xt = row_x<InT>(kp, ri, token, sh);
        lp_write(kp, r, sh.lp_list, c, m, ri.s2o, log2f(float(zt)), xt);
    }
    __syncthreads();
}

// ---------------------------------------------------------------- one unit
// A unit with an extension, once its copy has landed: staged whole (the vectors
// the bulk copy left out, a ragged tail or an unaligned slice, are loaded into
// the slot, which holds the whole unit), then rewritten in place: the mask
// (mws: the unit's mask words, word 0 holding token c0) turns disallowed tokens
// to -inf, and so do the nx biased and banned tokens xi (their values are taken
// apart). Out of line: the step without extensions keeps its code compact.
template <typename InT>
__device__ __noinline__ int stage_extensions(SliceView<InT> sv, bool masked, const uint32_t* mws,
                                             const int32_t* xi, int nx)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const int c0 = sv.c0;
    uint4* smv = const_cast<uint4*>(sv.sm);
    if (sv.nb < sv.nvec) {
        for (int j = sv.nb + lane; j < sv.nvec; j += 32) smv[j] = sv.vec(j);
        sv.nb = sv.nvec;
    }
    __syncwarp();
    if (masked) {
#pragma unroll 4
        for (int j = lane; j < sv.nb; j += 32) {
            const int t = j * E + (c0 & 31);
            const uint32_t bits = (mws[t >> 5] >> (t & 31)) & ((1u << E) - 1u);
            if (bits != (1u << E) - 1u) smv[j] = Vec<InT>::masked(smv[j], bits);
        }
        __syncwarp();
    }
    if (nx) {
        uint32_t* smw = reinterpret_cast<uint32_t*>(smv);
        for (int i = lane; i < nx; i += 32) {
            const int o = xi[i] - c0;
            if (sizeof(InT) == 2) {
                const int sh = 16 * (o & 1);
                atomicOr(&smw[o >> 1], 0xFF80u << sh);
                atomicAnd(&smw[o >> 1], ~(0x007Fu << sh));
            } else {
                smw[o] = 0xFF800000u;
            }
        }
        __syncwarp();
    }
    return sv.nb;
}

// Wait for the warp's slot, summarise the unit into its record (row r, slice s).
// Returns false, with nothing recorded, when the row's parameters are bad.
template <typename InT>
__device__ __forceinline__ bool process_unit(const SliceParams& P, const RowInfo& ri, uint64_t* bar,
                                             const unsigned char* slot, uint16_t* q, uint4* qw, int32_t* xi,
                                             float* xv, uint32_t parity, int r, int s, uint32_t off_lo,
                                             uint32_t off_hi)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const KernelParams& kp = P.k;
    const int G = P.G;
    const int c0 = s * P.W;
    const int n_el = min(P.W, int(kp.vocab) - c0);
    // While the copy is in flight: the unit's biased and banned tokens with
    // their final values (logit_bias / min_tokens), and its vocabulary-mask
    // words (into the queue scratch, free until the summary).
    int nx = 0;
    uint32_t* mws = reinterpret_cast<uint32_t*>(q);
    if (ri.cls != kClsErr) {
        if (has_extras(kp)) nx = row_extras<InT>(kp, ri, c0, c0 + n_el, xi, xv);
        if (mask_of(kp) && nx >= 0) {
            const uint32_t* mrow = mask_of(kp) + size_t(r) * size_t(kp.mask_stride) + (c0 >> 5);
            const int nw = ((c0 + n_el - 1) >> 5) - (c0 >> 5) + 1;
            uint32_t w[kMaskWords / 32];
#pragma unroll
            for (int i = 0; i < kMaskWords / 32; ++i) w[i] = 32 * i + lane < nw ? __ldg(mrow + 32 * i + lane) : 0u;
#pragma unroll
            for (int i = 0; i < kMaskWords / 32; ++i)
                if (32 * i + lane < nw) mws[32 * i + lane] = w[i];
        }
    }
    uint32_t extra = 0;
    // when the wait gives up, the unit is marked and the copy is still awaited
    // (with a longer bound) before the slot is reused
    if (!mbar_wait_bounded(bar, parity, P.max_polls)) {
        extra = kFlagTimeout;
        mbar_wait_bounded(bar, parity, kDrainPolls);
    }
    SLC_MARK(3);
    if (ri.cls == kClsErr || nx < 0) return false;
    SliceView<InT> sv;
    sv.sm = reinterpret_cast<const uint4*>(slot);
    sv.g = slice_ptr<InT>(kp, ri.lrow, c0);
    sv.nb = bulk_vecs<InT>(sv.g, n_el);
    sv.nvec = (n_el + E - 1) / E;
    sv.n = n_el;
    sv.c0 = c0;
    // The extensions rewrite the unit in place, so a unit that has one is staged
    // whole: the vectors the bulk copy left out (a ragged tail, an unaligned
    // slice) are loaded into the slot too (it holds the whole unit). NaN
    // sanitising is left to the first lane-maximum pass (a lane that meets a
    // NaN cleans its vectors).
    if (!extra && (sanitizing(kp) || mask_of(kp) || nx > 0)) {
        sv.nb = stage_extensions<InT>(sv, mask_of(kp) != nullptr, mws, xi, nx);
        sv.san = sanitizing(kp);
    }
    SliceHdr hdr;
    hdr.mx = -INFINITY;
    hdr.amax = INT_MAX;
    hdr.flags = kFlagAnyFinite;  // a unit that gave up reports only the timeout
    hdr.n = 0;
    K2 g{0ull, 0ull};
    SliceBody* body = P.body + size_t(r) * G + s;
    if (!extra) {
        if (ri.cls == kClsGreedy) {
            float lm;
            unit_max<InT>(sv, hdr.mx, hdr.amax, hdr.flags, lm);
            if (nx) {
                hdr.flags |= extras_flags(xv, nx);
                extras_max(xi, xv, nx, hdr.mx, hdr.amax);
            }
            if (row_lp(ri)) unit_trunc<InT>(sv, ri, hdr, body, reinterpret_cast<uint32_t*>(q), xi, xv, nx);
        } else if (ri.cls == kClsPlain) {
            unit_plain<InT>(sv, ri, off_lo, off_hi, q, qw, g, hdr.flags);
            if (nx) {  // the biased tokens, scored exactly
                hdr.flags |= extras_flags(xv, nx);
                const RowPhilox rp = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, off_lo, off_hi);
                K2 t{0ull, 0ull};
                for (int i = lane; i < nx; i += 32)
                    if (xv[i] > -INFINITY && xv[i] < INFINITY)
                        k2_insert(t, gkey(score2(xv[i], ri.s2, philox_word(rp, xi[i])), xi[i]));
                k2_warp_reduce(t);
                if (t.a) k2_insert(g, t.a);
                if (t.b) k2_insert(g, t.b);
            }
            __syncwarp();
            if (row_lp(ri)) unit_trunc<InT>(sv, ri, hdr, body, reinterpret_cast<uint32_t*>(q), xi, xv, nx);
        } else {
            unit_trunc<InT>(sv, ri, hdr, body, reinterpret_cast<uint32_t*>(q), xi, xv, nx,
                            P.cnt + size_t(r) * kCntStride + kHistOff);
        }
    }
    hdr.flags |= extra;
    if (lane == 0) {
        *reinterpret_cast<uint4*>(P.hdr + size_t(r) * G + s) =
            make_uint4(__float_as_uint(hdr.mx), uint32_t(hdr.amax), hdr.flags, hdr.n);
        if (ri.cls == kClsPlain)
            *reinterpret_cast<uint4*>(&body->ga) =
                make_uint4(uint32_t(g.a), uint32_t(g.a >> 32), uint32_t(g.b), uint32_t(g.b >> 32));
    }
    return true;
}

// Finish row r (this warp's arrival completed it), and its logprob outputs when
// they are asked; scratch: the warp's idle staging slot. Returns false when the
// row is left for the exact path (m: the row maximum).
template <typename InT>
__device__ SLC_FIN_INLINE bool finish_row(const SliceParams& P, WarpScratch& ws, const RowInfo& ri, int r,
                                        uint32_t off_lo, uint32_t off_hi, unsigned char* scratch, float& m)
{
    m = -INFINITY;
    int tok = -1;
    int32_t st = 0;
    if (ri.cls == kClsGreedy) {
        finish_greedy(P, r, tok, st);
    } else if (ri.cls == kClsPlain) {
        finish_plain<InT>(P, ri, r, off_lo, off_hi, tok, st);
    } else if (!finish_trunc<InT>(P, ws, ri, r, off_lo, off_hi, scratch, m, tok, st)) {
        return false;
    }
    // outputs over the whole row (untruncated rows; every row when unscaled)
    if (row_lp(ri) && (P.k.lp_unscaled || ri.cls != kClsTrunc)) {
        __syncwarp();
        return finish_lp_row<InT>(P, ws, ri, r, tok, st, scratch, m);
    }
    return true;
}

// ---------------------------------------------------------------- the kernel
template <typename InT>
__global__ void __launch_bounds__(kT, 1) slice_kernel(const __grid_constant__ SliceParams P)
{
    extern __shared__ __align__(128) unsigned char smem[];
    SliceShared& sh = *reinterpret_cast<SliceShared*>(smem);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    WarpScratch& ws = sh.ws[wid];
    const KernelParams& kp = P.k;
    const int NC = int(gridDim.x);
    const int stride = NC * kW;
    SLC_MARK(0);
    // slot s of the CTA stages its units blockIdx.x + s * NC (+ k * stride):
    // round-robin over CTAs first. The copy of its first unit goes out before
    // anything else, unless the kernel is the programmatic dependent of the
    // grid that writes the logits: then it goes out once that grid is done,
    // after the set-up below.
    const int u0 = int(blockIdx.x) + wid * NC;
    if (lane == 0) {
        mbar_init(&sh.full[wid], 1);
        fence_mbar_init();
        if (!P.pdl && u0 < P.n_units) issue_unit<InT>(P, &sh.full[wid], smem + kHead + size_t(wid) * kSlotBytes, u0);
    }
    if (tid == 0) sh.n_exact = 0;
    const uint64_t off = kp.philox_offset_dev ? *kp.philox_offset_dev : kp.philox_offset;
    const uint32_t off_lo = uint32_t(off), off_hi = uint32_t(off >> 32);
    // which slot this warp serves: the CTA's first units, by their cost (plain
    // rows far above truncated ones, those above greedy ones), dealt over the
    // four schedulers (warp w runs on scheduler w % 4) in snake order
    int sidx;
    RowInfo ri0;  // the parameters of the row of the slot's first unit
    {
        const int ul = int(blockIdx.x) + (lane & (kW - 1)) * NC;
        int cost = 0;
        RowInfo mine{};
        if (ul < P.n_units) {
            mine = load_info(P, ul / P.G);
            const uint8_t c = mine.cls;
            cost = c == kClsPlain ? 3 : c == kClsTrunc ? 2 : c == kClsGreedy ? 1 : 0;
        }
        // rank among the 16 (cost descending, slot ascending)
        int rank = 0;
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t same = __ballot_sync(0xffffffffu, lane < kW && cost == c);
            rank += c > cost ? __popc(same) : c == cost ? __popc(same & lt) : 0;
        }
        const int row4 = rank >> 2, col = rank & 3;
        const int w_of = row4 * 4 + ((row4 & 1) ? 3 - col : col);
        const uint32_t hit = __ballot_sync(0xffffffffu, lane < kW && w_of == wid);
        sidx = __ffs(hit) - 1;
        uint32_t wmine[sizeof(RowInfo) / 4], w0[sizeof(RowInfo) / 4];
        memcpy(wmine, &mine, sizeof(RowInfo));
#pragma unroll
        for (int q = 0; q < int(sizeof(RowInfo) / 4); ++q) w0[q] = __shfl_sync(0xffffffffu, wmine[q], sidx);
        memcpy(&ri0, w0, sizeof(RowInfo));
    }
    if (P.pdl) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (lane == 0 && u0 < P.n_units)
            issue_unit<InT>(P, &sh.full[wid], smem + kHead + size_t(wid) * kSlotBytes, u0);
    }
    unsigned char* slot = smem + kHead + size_t(sidx) * kSlotBytes;
    uint64_t* bar = &sh.full[sidx];
    int u = int(blockIdx.x) + sidx * NC;
    __syncthreads();  // barriers initialised, n_exact set before any warp can queue a row
    SLC_MARK(1);
    uint32_t parity = 0;
    bool first = true;
#pragma unroll 1
    while (u < P.n_units) {
        const int r = u / P.G, s = u - r * P.G;
        const RowInfo ri = first ? ri0 : load_info(P, r);
        first = false;
        SLC_MARK(2);
        SLC_UCLS(ri.cls);
        const bool ok = process_unit<InT>(P, ri, bar, slot, ws.q, ws.qw, ws.xi, ws.xv, parity, r, s, off_lo, off_hi);
        SLC_MARK(5);
        parity ^= 1u;
        const int un = u + stride;
        if (!ok) {
            if (s == 0 && lane == 0) write_out(kp, r, -1, kRowBadParam);
        } else {
            // the arrival is a release (publishing this unit's record) and an acquire
            // (seeing every other unit's record when it completes the row)
            __syncwarp();
            uint32_t old = 0;
            if (lane == 0) old = atom_add_acq_rel(&P.cnt[size_t(r) * kCntStride], 1u);
            old = __shfl_sync(0xffffffffu, old, 0);
            SLC_MARK(6);
            if (old == uint32_t(P.G - 1)) {
                __syncwarp();
                float m;
                SLC_TAG(ri.cls);
                const bool done = finish_row<InT>(P, ws, ri, r, off_lo, off_hi, slot, m);
                SLC_MARK(12);
                if (lane == 0) {
                    P.cnt[size_t(r) * kCntStride] = 0;
                    if (!done) {
                        const int q = atomicAdd(&sh.n_exact, 1);
                        sh.exact_rows[q] = r;
                        sh.exact_m[q] = m;
                    }
                }
            }
        }
        // the slot is free (also of any finishing scratch): the next unit's copy
        __syncwarp();
        if (lane == 0 && un < P.n_units) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_unit<InT>(P, bar, slot, un);
        }
        u = un;
    }
    SLC_MARK(13);
    // rows the candidate lists could not settle
    __syncthreads();
    const int ne = sh.n_exact;
    for (int q = 0; q < ne; ++q) {
        const int r = sh.exact_rows[q];
        cta_exact_row<InT>(sh, smem + kHead, P, r, load_info(P, r), sh.exact_m[q], off_lo, off_hi);
    }
}

}  // namespace SLC_VARIANT
}  // namespace slc
}  // namespace dst
