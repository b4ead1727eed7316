// slice_sampler.cuh -- the slice kernel: small batches without history or
// probs / logprobs outputs (sm_103a).
//
// Layout of the work. Each row is cut into G equal slices of W elements (at
// most one warp's staging slot); a (row, slice) pair is a unit, and the units
// are dealt round-robin over the CTAs first and then over the warps of each
// CTA, so that the 16 warps of an SM hold slices of 16 different rows. On the
// 64-row, 128000-token batch this is exactly one unit per warp of the GPU.
// Every warp works on its own:
//
//   staging   lane 0 arms the warp's mbarrier and starts one 1-D bulk
//             (TMA-engine) copy of the unit into the warp's shared-memory slot
//             before anything else, so the whole batch is requested at once;
//             the row's parameters are read while the copy flies.
//   summary   the warp summarises its unit into a record in global memory:
//               greedy     the unit maximum and its lowest index;
//               plain      the unit's best two Gumbel scores x/T - ln E. Each
//                          lane scores its largest logit exactly; the second
//                          best of these 32 scores bounds the unit's second
//                          best from below, and a per-token bound
//                          x/T - ln(1 - u) (one MUFU log2) against it leaves
//                          almost no token to score exactly;
//               truncated  the unit maximum, its largest lane maxima (a sketch
//                          of up to 8 order keys: at least that many tokens
//                          reach each of them), tau = the smallest of them, and
//                          every token at or above tau (a short list, complete
//                          above tau).
//   arrival   an acquire-release atomic add on the row's counter (one counter
//             per 128-byte line); the warp whose arrival completes the row
//             finishes it at once and resets the counter. Nothing ever waits
//             on another warp.
//   finish    greedy and plain rows reduce their G records. A truncated row
//             takes a bound B at or below every kept token (top-k: the k-th
//             largest sketch key over the row, a 16-bit prefix found by a
//             two-level histogram; min-p: the threshold), gathers the listed
//             tokens >= B, reads again from global memory the slices whose
//             lists are not complete above B, sorts the candidates and cuts
//             top-k, top-p and min-p before the Gumbel pick. Rows the lists
//             cannot settle (top-k above 128, a top-p cut beyond the lists,
//             too many candidates) are sampled by the whole CTA after its warps
//             are done, streaming the row.
//
// Stage order and definitions follow the xbrilliance.ai note "采样参数对解码开销的影响：
// temperature、top_p 与采样核路径", section "解码一步里采样做什么" (penalties,
// temperature, top-k / top-p, min-p, softmax, pick), and the Gumbel-max rule of
// the dev.to claim check "SGLang's +75% sampler speedup skips Qwen3 chat
// requests", section "Nine lines, and exactly one call site".
#pragma once

#include <cuda_bf16.h>

#include <cfloat>
#include <climits>
#include <cstdint>

#include "row_sampler.cuh"

namespace dst {
namespace slc {

constexpr int kT = 512;                 // threads per CTA
constexpr int kW = kT / 32;             // warps per CTA
constexpr int kMaxRows = 256;           // rows the slice kernel takes
constexpr int kMaxSlices = 128;         // slices per row
constexpr int kSPL = kMaxSlices / 32;   // slices per lane when finishing
constexpr int kSketch = 8;              // lane maxima a truncated unit exposes
constexpr int kLCap = 48;               // list entries one record holds
constexpr int kKComplete = 32;          // top-k rows up to this k list each unit's top k
constexpr int kMaxTopN = 16;            // largest top_n of the logprob outputs
constexpr int kMaxBias = 64;            // logit_bias entries a row may carry
constexpr int kMaxStop = 16;            // stop tokens a row may carry (min_tokens)
constexpr int kMaxExtras = kMaxBias + kMaxStop;  // tokens taken apart from the staged logits
constexpr int kTQCap = 320;             // vectors a truncated unit queues (more: the list overflows)
constexpr int kKCap = 128;              // largest top-k the lists settle
constexpr int kReCap = 16;              // slices a finishing warp may read again
constexpr int kRankSortMax = 256;       // candidates sorted by counting ranks (more: bitonic)
constexpr int kSlotBytes = 10240;       // a warp's staging slot
constexpr int kMinUnit = 2048;          // smallest unit, in elements (unless the row is narrower)
constexpr int kMaskWords = (kSlotBytes / 2 / 32 + 2 + 31) / 32 * 32;  // mask words a unit spans, rounded up to 32
constexpr uint32_t kOverflow = 0xFFFFFFFFu;
constexpr uint32_t kDrainPolls = 1u << 26;  // polls granted to a copy after a wait gave up
// Each row's arrival counter sits in its own 128-byte line: G warps add to every
// counter, and counters sharing a line would serialise their atomics in one L2
// slice.
constexpr int kCntStride = 32 + 256;  // per row: the arrival counter's line, then the sketch-key histogram
constexpr int kHistOff = 32;          // first histogram word
constexpr int kHistBins = 256;        // bins of 1/4 over the logits [-32, 32) (the outer two take the rest)

enum : uint8_t { kClsTrunc = 0, kClsPlain = 1, kClsGreedy = 2, kClsErr = 3 };

// One (row, slice) summary in global memory.
struct alignas(16) SliceHdr {
    float mx;       // unit maximum (NaN ignored), -inf when nothing is finite
    int32_t amax;   // its lowest index
    uint32_t flags; // kFlag* bits
    uint32_t n;     // truncated rows: listed tokens, kOverflow when they did not fit
};

struct alignas(16) SliceBody {
    // plain rows: the unit's best two Gumbel scores as composite keys (order key
    // of the fp32 score << 32 | ~token: larger is better, ties to the lower
    // token), 0 when absent
    unsigned long long ga, gb;
    uint32_t tau;   // truncated rows: order key every listed token reaches
    float zs;       // top-p rows without top-k: sum of exp((x - mx) / T) over the unit
    float zc;       // its low-order part (the sum is zs + zc)
    uint32_t m;     // entries of the sketch
    float zos;      // logprob outputs over the whole row: sum of exp((x - mx) / T_out)
    float zoc;      // its low-order part
    uint32_t zpad0, zpad1;
    uint32_t sketch[kSketch];        // truncated rows: largest lane maxima (order keys, descending)
    unsigned long long list[kLCap];  // truncated rows: cand_word of each listed token
};

struct SliceParams {
    KernelParams k;
    int32_t n_rows;
    int32_t G;           // slices per row
    int32_t W;           // elements per slice (a multiple of 16 bytes)
    int32_t n_units;     // n_rows * G
    SliceHdr* hdr;       // [n_rows][G]
    SliceBody* body;     // [n_rows][G]
    uint32_t* cnt;       // [n_rows * kCntStride] arrivals (one per line) and sketch-key histograms; zero between launches
    unsigned long long* stats;  // [0]: rows finished by the exact path (may be NULL)
    uint32_t max_polls;  // bound of each wait on a staging copy
    int32_t pdl;         // launched as a programmatic dependent: wait for the grid before it
};

struct alignas(16) RowInfo {
    float T;       // temperature used for scores (1 for greedy rows)
    float invT;
    float s2;      // log2(e) / T: scores are kept in log2 units
    float p, minp;
    int32_t k;
    uint32_t stream, key_lo, key_hi;
    int32_t lrow;
    float s2o;     // log2(e) / T of the logprob outputs (1 when unscaled)
    uint8_t cls, do_topk, do_topp, do_minp;
    uint8_t need_z, m, mt, greedy;
    uint8_t lp;    // logprob outputs requested
    uint8_t need_zo;  // the units keep the row's softmax mass at the outputs' temperature
    uint8_t ban;   // min_tokens: the row's stop tokens are -inf
    uint8_t pad3;
    int32_t r;     // the output row
};

struct alignas(16) WarpScratch {
    uint16_t q[kSlotBytes / 16];        // plain units: vectors the cheap bound let through;
                                        // truncated units: (vector << 8 | mask) words
    uint4 qw[2 * 32];                   // Philox words of the first 32 queued vectors
    int32_t xi[kMaxExtras];             // logit_bias / min_tokens: the unit's biased and
    float xv[kMaxExtras];               // banned tokens, and their final logits
    uint32_t n;                         // candidates listed
    uint32_t nre;                       // slices to read again
    uint16_t re[kReCap];
};

struct alignas(16) SliceShared {
    uint64_t full[kW];            // one staging mbarrier per warp
    WarpScratch ws[kW];
    int32_t n_exact;
    int32_t exact_rows[kMaxRows]; // rows left for the CTA's exact path
    float exact_m[kMaxRows];
    // CTA-wide scratch of the exact path
    uint32_t hcnt[256];
    unsigned long long hmass[256];
    unsigned long long scan_w[kW];
    int32_t red_i[kW];
    unsigned long long red_k[2 * kW];
    unsigned long long sel_prefix, sel_wabove, sel_target;
    double red_d[kW];
    // logit_bias / min_tokens on the exact path: the row's biased and banned
    // tokens, their values, and a bitmap of them (in the idle staging slots)
    int32_t bx_i[kMaxExtras];
    float bx_v[kMaxExtras];
    int32_t bx_n;
    uint32_t* bx_bits;
    unsigned long long lp_list[kMaxTopN];
    int32_t lp_cnt;
    int32_t sel_idx;
    int32_t pad;
};

constexpr size_t kHead = (sizeof(SliceShared) + 127) & ~size_t(127);
constexpr size_t kSmemBytes = kHead + size_t(kW) * kSlotBytes;
constexpr size_t kMaxSmem = 227 * 1024;
static_assert(kSmemBytes <= kMaxSmem, "shared memory per CTA");
static_assert(kSlotBytes >= 1024 * 8, "a free slot holds 1024 candidates");
static_assert(kMaxSlices * 64 + kHistBins * 4 <= kSlotBytes, "a truncated row's finish stages its records and histogram in a slot");
static_assert(kTQCap * 4 <= int(sizeof(WarpScratch::q)) && kTQCap > kLCap, "truncated-unit queue");
static_assert(kMaskWords * 4 <= int(sizeof(WarpScratch::q)) && kMaskWords >= kSlotBytes / 2 / 32 + 2,
              "a unit's mask words fit the queue scratch");

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ void warp_max_idx(float& m, int& i)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, off);
        const int oi = __shfl_xor_sync(0xffffffffu, i, off);
        if (om > m || (om == m && oi < i)) {
            m = om;
            i = oi;
        }
    }
}

// The 8 (bf16) or 4 (fp32) logits of a 16-byte vector.
template <typename InT>
struct Vec;

template <>
struct Vec<uint16_t> {
    static constexpr int E = 8;
    __device__ static __forceinline__ float get(const uint4& r, int e) { return ElemTraits<uint16_t>::get(r, e); }
    // running maximum in packed form, NaN-propagating (four bf16x2 lanes)
    __device__ static __forceinline__ uint4 neg_inf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
    // elements whose bit is clear become -inf
    __device__ static __forceinline__ uint32_t mask_word(uint32_t w, uint32_t b2)
    {
        const uint32_t keep = ((b2 & 1u) ? 0x0000FFFFu : 0u) | ((b2 & 2u) ? 0xFFFF0000u : 0u);
        return (w & keep) | (0xFF80FF80u & ~keep);
    }
    __device__ static __forceinline__ uint4 masked(const uint4& v, uint32_t bits)
    {
        return make_uint4(mask_word(v.x, bits), mask_word(v.y, bits >> 2), mask_word(v.z, bits >> 4),
                          mask_word(v.w, bits >> 6));
    }
    // NaN elements become -inf
    __device__ static __forceinline__ uint32_t sanitize_word(uint32_t w)
    {
        const uint32_t nan = (((w & 0x7FFFu) > 0x7F80u) ? 0x0000FFFFu : 0u) |
                             (((w & 0x7FFF0000u) > 0x7F800000u) ? 0xFFFF0000u : 0u);
        return (w & ~nan) | (0xFF80FF80u & nan);
    }
    __device__ static __forceinline__ uint4 sanitized(const uint4& v)
    {
        return make_uint4(sanitize_word(v.x), sanitize_word(v.y), sanitize_word(v.z), sanitize_word(v.w));
    }
    using Acc = uint4;
    __device__ static __forceinline__ Acc acc_init() { return neg_inf(); }
    __device__ static __forceinline__ uint32_t hmax_nan(uint32_t a, uint32_t b)
    {
        const __nv_bfloat162 r = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                             *reinterpret_cast<const __nv_bfloat162*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
    __device__ static __forceinline__ void acc_add(Acc& a, const uint4& v)
    {
        a.x = hmax_nan(a.x, v.x);
        a.y = hmax_nan(a.y, v.y);
        a.z = hmax_nan(a.z, v.z);
        a.w = hmax_nan(a.w, v.w);
    }
    // the maximum, or NaN when one was seen
    __device__ static __forceinline__ float acc_max(const Acc& a)
    {
        const uint32_t m = hmax_nan(hmax_nan(a.x, a.y), hmax_nan(a.z, a.w));
        const float lo = __uint_as_float(m << 16), hi = __uint_as_float(m & 0xFFFF0000u);
        return (lo != lo || hi != hi) ? __uint_as_float(0x7FFFFFFFu) : fmaxf(lo, hi);
    }
    __device__ static __forceinline__ __nv_bfloat162 bf2(uint32_t w)
    {
        __nv_bfloat162 r;
        memcpy(&r, &w, 4);
        return r;
    }
    // whether some element equals m (a non-NaN bf16 value; -0 equals +0)
    __device__ static __forceinline__ bool has(const uint4& v, float m)
    {
        const __nv_bfloat162 m2 = __float2bfloat162_rn(m);
        return (__heq2_mask(bf2(v.x), m2) | __heq2_mask(bf2(v.y), m2) | __heq2_mask(bf2(v.z), m2) |
                __heq2_mask(bf2(v.w), m2)) != 0u;
    }
    // elements >= t (a bf16 value), as two 16-bit counts in one word: add the
    // words of up to 16383 vectors, then fold them with count_fold
    using Thr = __nv_bfloat162;
    __device__ static __forceinline__ Thr thr(float t) { return __float2bfloat162_rn(t); }
    __device__ static __forceinline__ uint32_t count_ge(const uint4& v, Thr t2)
    {
        return (__hge2_mask(bf2(v.x), t2) & 0x10001u) + (__hge2_mask(bf2(v.y), t2) & 0x10001u) +
               (__hge2_mask(bf2(v.z), t2) & 0x10001u) + (__hge2_mask(bf2(v.w), t2) & 0x10001u);
    }
    __device__ static __forceinline__ uint32_t count_fold(uint32_t c) { return (c & 0xFFFFu) + (c >> 16); }
    // bit e set when element e >= t
    __device__ static __forceinline__ uint32_t mask_ge(const uint4& v, Thr t2)
    {
        const uint32_t m0 = __hge2_mask(bf2(v.x), t2), m1 = __hge2_mask(bf2(v.y), t2);
        const uint32_t m2 = __hge2_mask(bf2(v.z), t2), m3 = __hge2_mask(bf2(v.w), t2);
        return ((m0 & 1u) | ((m0 >> 15) & 2u)) | (((m1 & 1u) | ((m1 >> 15) & 2u)) << 2) |
               (((m2 & 1u) | ((m2 >> 15) & 2u)) << 4) | (((m3 & 1u) | ((m3 >> 15) & 2u)) << 6);
    }
};

template <>
struct Vec<float> {
    static constexpr int E = 4;
    __device__ static __forceinline__ float get(const uint4& r, int e) { return ElemTraits<float>::get(r, e); }
    __device__ static __forceinline__ uint4 neg_inf() { return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u); }
    __device__ static __forceinline__ uint4 masked(const uint4& v, uint32_t bits)
    {
        return make_uint4((bits & 1u) ? v.x : 0xFF800000u, (bits & 2u) ? v.y : 0xFF800000u,
                          (bits & 4u) ? v.z : 0xFF800000u, (bits & 8u) ? v.w : 0xFF800000u);
    }
    __device__ static __forceinline__ uint32_t sanitize_word(uint32_t w)
    {
        return (w & 0x7FFFFFFFu) > 0x7F800000u ? 0xFF800000u : w;
    }
    __device__ static __forceinline__ uint4 sanitized(const uint4& v)
    {
        return make_uint4(sanitize_word(v.x), sanitize_word(v.y), sanitize_word(v.z), sanitize_word(v.w));
    }
    using Acc = float4;
    __device__ static __forceinline__ Acc acc_init() { return make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY); }
    __device__ static __forceinline__ float fmax_nan(float a, float b)
    {
        float r;
        asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
        return r;
    }
    __device__ static __forceinline__ void acc_add(Acc& a, const uint4& v)
    {
        a.x = fmax_nan(a.x, __uint_as_float(v.x));
        a.y = fmax_nan(a.y, __uint_as_float(v.y));
        a.z = fmax_nan(a.z, __uint_as_float(v.z));
        a.w = fmax_nan(a.w, __uint_as_float(v.w));
    }
    __device__ static __forceinline__ float acc_max(const Acc& a)
    {
        return fmax_nan(fmax_nan(a.x, a.y), fmax_nan(a.z, a.w));
    }
    __device__ static __forceinline__ bool has(const uint4& v, float m)
    {
        return __uint_as_float(v.x) == m || __uint_as_float(v.y) == m || __uint_as_float(v.z) == m ||
               __uint_as_float(v.w) == m;
    }
    using Thr = float;
    __device__ static __forceinline__ Thr thr(float t) { return t; }
    __device__ static __forceinline__ uint32_t count_ge(const uint4& v, Thr t)
    {
        return uint32_t(__uint_as_float(v.x) >= t) + uint32_t(__uint_as_float(v.y) >= t) +
               uint32_t(__uint_as_float(v.z) >= t) + uint32_t(__uint_as_float(v.w) >= t);
    }
    __device__ static __forceinline__ uint32_t count_fold(uint32_t c) { return c; }
    __device__ static __forceinline__ uint32_t mask_ge(const uint4& v, Thr t)
    {
        return uint32_t(__uint_as_float(v.x) >= t) | (uint32_t(__uint_as_float(v.y) >= t) << 1) |
               (uint32_t(__uint_as_float(v.z) >= t) << 2) | (uint32_t(__uint_as_float(v.w) >= t) << 3);
    }
};

// One unit as a warp sees it: staged vectors [0, nb) in shared memory, the rest
// (a ragged tail, or everything for a slice that is not 16-byte aligned) read
// from global memory, padded with -inf.
template <typename InT>
struct SliceView {
    const uint4* sm;
    const InT* g;    // first element of the slice in global memory
    int nb;          // staged vectors (with the row's extensions applied)
    int nvec;        // vectors covering the slice
    int n;           // elements in the slice
    int c0;          // first token of the slice
    bool san = false;  // NaN sanitising: the first lane-maximum pass cleans the (whole) staged unit

    __device__ __forceinline__ uint4 vec(int j) const
    {
        if (j < nb) return sm[j];
        constexpr int E = Vec<InT>::E;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < E; ++q) {
            const int i = j * E + q;
            if (sizeof(InT) == 2) {
                const uint32_t b = i < n ? uint32_t(reinterpret_cast<const uint16_t*>(g)[i]) : 0xFF80u;
                if (q & 1) w[q >> 1] |= b << 16;
                else w[q >> 1] = b;
            } else {
                w[q] = i < n ? reinterpret_cast<const uint32_t*>(g)[i] : 0xFF800000u;
            }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

__device__ __forceinline__ uint32_t flags_of(bool nan, float vmax)
{
    uint32_t f = 0;
    if (nan || vmax == INFINITY) f |= kFlagNonFinite;
    if (vmax > -INFINITY && vmax < INFINITY) f |= kFlagAnyFinite;
    return f;
}

__device__ __forceinline__ uint32_t warp_or(uint32_t v) { return __reduce_or_sync(0xffffffffu, v); }

// Exact Gumbel score in log2 units: log2(e) * (x / T - ln E). Out of line so
// that every caller shares one copy of the code.
static __device__ __noinline__ float score2(float x, float s2, uint32_t w)
{
    return x * s2 - log2f(noise_exp1_f32(w));
}

// ---------------------------------------------------------------- composite keys
// A Gumbel candidate as one 64-bit word: order key of its fp32 score (log2
// units) above the complemented token, so that max() ranks by score and breaks
// ties to the lower token; 0 is "none".
__device__ __forceinline__ unsigned long long gkey(float s, int v) { return cand_word(f2key(s), v); }
__device__ __forceinline__ float gkey_score(unsigned long long c) { return key2f(cand_key(c)); }

struct K2 {
    unsigned long long a, b;  // a >= b
};

__device__ __forceinline__ void k2_insert(K2& t, unsigned long long c)
{
    if (c > t.a) {
        t.b = t.a;
        t.a = c;
    } else if (c > t.b) {
        t.b = c;
    }
}

// Best two of the warp (every lane gets them).
__device__ __forceinline__ void k2_warp_reduce(K2& t)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long oa = __shfl_xor_sync(0xffffffffu, t.a, off);
        const unsigned long long ob = __shfl_xor_sync(0xffffffffu, t.b, off);
        const bool mine = t.a >= oa;
        const unsigned long long lo = mine ? oa : t.a;   // the smaller of the two firsts
        const unsigned long long sec = mine ? t.b : ob;  // the winner's second
        t.a = mine ? t.a : oa;
        t.b = lo > sec ? lo : sec;
    }
}

// Bound on the fp32 error of the difference of two scores score2() returns:
// when two scores differ by more, their order is the order of the exact
// (double-precision) scores.
__device__ __forceinline__ float settle_eps(float sa, float sb)
{
    return 3e-5f + 1e-6f * (fabsf(sa) + fabsf(sb));
}

}  // namespace slc
}  // namespace dst
