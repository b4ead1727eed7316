// slice_kernel.cuh -- body of the slice kernel (design in slice_sampler.cuh).
//
// Every warp runs on its own: its unit's copy, its row's parameters, its
// summary, its arrival and, when it completes a row, that row's finish. The
// only CTA-wide step is the exact path at the end, for rows the candidate
// lists could not settle.
#pragma once

#include "slice_sampler.cuh"

namespace dst {
namespace slc {

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
    const bool greedy = T < 1e-5f;
    ri.T = greedy ? 1.0f : T;
    ri.invT = 1.0f / ri.T;
    ri.s2 = 1.4426950408889634f / ri.T;
    ri.do_topk = (ri.k != -1 && int64_t(ri.k) < V);
    ri.do_topp = ri.p < 1.0f;
    ri.do_minp = ri.minp > 0.0f;
    ri.need_z = ri.do_topp && !ri.do_topk;
    ri.m = uint8_t(ri.do_topk ? min(ri.k, kSketch) : kSketch);
    ri.pad0 = ri.pad1 = 0;
    if (bad) ri.cls = kClsErr;
    else if (greedy) ri.cls = kClsGreedy;
    else if (!ri.do_topk && !ri.do_topp && !ri.do_minp) ri.cls = kClsPlain;
    else ri.cls = kClsTrunc;
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

// Lane maximum (NaN ignored), its lowest token, and the flags of the part of
// the unit a lane reads.
template <typename InT>
__device__ __forceinline__ void lane_max(const SliceView<InT>& sv, float& m, int& mi, uint32_t& f)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    m = -INFINITY;
    mi = INT_MAX;
    f = 0;
#pragma unroll 1
    for (int j = lane; j < sv.nvec; j += 32) {
        const uint4 v = sv.vec(j);
        bool nan;
        const float vm = Vec<InT>::vmax(v, nan);
        f |= flags_of(nan, vm);
        if (vm > m) {
            m = vm;
            mi = sv.c0 + j * E + vec_find<InT>(v, vm);
        }
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

template <typename InT>
__device__ __forceinline__ void unit_plain(const SliceView<InT>& sv, const RowInfo& ri, uint32_t off_lo,
                                           uint32_t off_hi, K2& out, uint32_t& flags)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    // each lane scores its largest logit exactly; the second-best of these 32
    // scores bounds the unit's second-best score from below
    float lm;
    int li;
    uint32_t f;
    lane_max<InT>(sv, lm, li, f);
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
    // every other token whose bound x/T - ln(1 - u) reaches thr (E >= 1 - u, so
    // the bound is at least the score; log2 units throughout)
#pragma unroll 1
    for (int j = lane; j < sv.nvec; j += 32) {
        const uint4 v = sv.vec(j);
        const int t0 = sv.c0 + j * E;
        uint4 b0, b1;
        vec_words<InT>(rp, t0, b0, b1);
        uint32_t hit = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float x = Vec<InT>::get(v, e);
            const uint32_t we = lane_of(e < 4 ? b0 : b1, uint32_t(e) & 3u);
            const float bound = fmaf(x, s2, -__log2f(noise_one_minus_u(we)));
            hit |= (bound >= thr ? 1u : 0u) << e;
        }
#pragma unroll 1
        for (; hit; hit &= hit - 1) {
            const int e = __ffs(hit) - 1;
            const int idx = t0 + e;
            const float x = Vec<InT>::get(v, e);
            if (idx == li || !(x > -INFINITY)) continue;
            const uint32_t we = lane_of(e < 4 ? b0 : b1, uint32_t(e) & 3u);
            k2_insert(t, gkey(score2(x, s2, we), idx));
        }
    }
    k2_warp_reduce(t);
    out = t;
}

// ---------------------------------------------------------------- truncated unit
template <typename InT>
__device__ __forceinline__ void unit_trunc(const SliceView<InT>& sv, const RowInfo& ri, SliceHdr& hdr_out,
                                           SliceBody* body)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    float lm;
    int li;
    uint32_t f;
    lane_max<InT>(sv, lm, li, f);
    const uint32_t flags = warp_or(f);
    float mx = lm;
    int amax = li;
    warp_max_idx(mx, amax);
    // the sketch: the m largest lane maxima (order keys, descending); tau is the
    // smallest of them, so at least m tokens reach tau
    const uint32_t lkey = lm > -INFINITY ? f2key(lm) : 0u;
    uint32_t left = lkey, tau = 0, m = 0;
#pragma unroll 1
    for (int q = 0; q < int(ri.m); ++q) {
        const uint32_t top = __reduce_max_sync(0xffffffffu, left);
        if (top == 0) break;
        tau = top;
        if (lane == 0) body->sketch[q] = top;
        ++m;
        const uint32_t holder = __ballot_sync(0xffffffffu, left == top);
        if (lane == __ffs(holder) - 1) left = 0;
    }
    tau = max(tau, 1u);  // -inf (key 0 here) is never listed
    // list every finite token whose key reaches tau: only lanes whose maximum
    // reaches it hold any
    uint32_t mine = 0;
    if (lkey >= tau) {
#pragma unroll 1
        for (int j = lane; j < sv.nvec; j += 32) {
            const uint4 v = sv.vec(j);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float x = Vec<InT>::get(v, e);
                mine += (x > -INFINITY && f2key(x) >= tau) ? 1u : 0u;
            }
        }
    }
    uint32_t incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t pos = incl - mine;
    if (mine && pos < uint32_t(kLCap)) {
#pragma unroll 1
        for (int j = lane; j < sv.nvec && pos < uint32_t(kLCap); j += 32) {
            const uint4 v = sv.vec(j);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float x = Vec<InT>::get(v, e);
                if (x > -INFINITY && f2key(x) >= tau) {
                    if (pos < uint32_t(kLCap)) body->list[pos] = cand_word(f2key(x), sv.c0 + j * E + e);
                    ++pos;
                }
            }
        }
    }
    // top-p rows without top-k: the unit's softmax mass at its maximum
    float zsum = 0.0f, zlow = 0.0f;
    if (ri.need_z && mx > -INFINITY && mx < INFINITY) {
        float zs = 0.0f, zc = 0.0f;  // Kahan: the sum is zs - zc
#pragma unroll 1
        for (int j = lane; j < sv.nvec; j += 32) {
            const uint4 v = sv.vec(j);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float x = Vec<InT>::get(v, e);
                if (!(x > -INFINITY)) continue;
                const float term = exp2f((x - mx) * ri.s2) - zc;
                const float sum = zs + term;
                zc = (sum - zs) - term;
                zs = sum;
            }
        }
        double z = double(zs) - double(zc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        zsum = float(z);
        zlow = float(z - double(zsum));
    }
    if (lane == 0)
        *reinterpret_cast<uint4*>(&body->tau) = make_uint4(tau, __float_as_uint(zsum), __float_as_uint(zlow), m);
    hdr_out.mx = mx;
    hdr_out.amax = amax;
    hdr_out.flags = flags;
    hdr_out.n = total > uint32_t(kLCap) ? kOverflow : total;
}

// ---------------------------------------------------------------- finishing
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

// The pick between the best two candidates in double precision (the exact
// Gumbel-max score); logits read again, Philox words recomputed.
template <typename InT>
__device__ __noinline__ int settle_pair(const KernelParams& kp, const RowInfo& ri, uint32_t off_lo, uint32_t off_hi,
                                        unsigned long long a, unsigned long long b)
{
    const int ia = cand_idx(a), ib = cand_idx(b);
    const RowPhilox rp = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, off_lo, off_hi);
    const float xa = ElemTraits<InT>::load(kp.logits, int64_t(ri.lrow) * kp.row_stride + ia);
    const float xb = ElemTraits<InT>::load(kp.logits, int64_t(ri.lrow) * kp.row_stride + ib);
    const double sa = gumbel_score_f64(xa, ri.T, philox_word(rp, ia));
    const double sb = gumbel_score_f64(xb, ri.T, philox_word(rp, ib));
    return (sa > sb || (sa == sb && ia < ib)) ? ia : ib;
}

// The pick from the best two candidates (composite keys; b may be 0): by their
// fp32 scores when those are further apart than their error bound, else in
// double precision.
template <typename InT>
__device__ __forceinline__ int pick_of(const KernelParams& kp, const RowInfo& ri, uint32_t off_lo, uint32_t off_hi,
                                       const K2& t)
{
    if (t.b == 0ull) return cand_idx(t.a);
    const float sa = gkey_score(t.a), sb = gkey_score(t.b);
    if (sa - sb > settle_eps(sa, sb)) return cand_idx(t.a);
    return settle_pair<InT>(kp, ri, off_lo, off_hi, t.a, t.b);
}

__device__ __forceinline__ void finish_greedy(const SliceParams& P, int r)
{
    const int lane = threadIdx.x & 31;
    const int G = P.G;
    const SliceHdr* hd = P.hdr + size_t(r) * G;
    float m = -INFINITY;
    int mi = INT_MAX;
    uint32_t fl = 0;
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        const int b = lane + 32 * i;
        if (b < G) {
            const SliceHdr h = ld_hdr(hd + b);
            fl |= h.flags;
            if (h.mx > m || (h.mx == m && h.amax < mi)) {
                m = h.mx;
                mi = h.amax;
            }
        }
    }
    fl = warp_or(fl);
    warp_max_idx(m, mi);
    if (lane == 0) write_out(P.k, r, mi, status_of(fl));
}

template <typename InT>
__device__ __forceinline__ void finish_plain(const SliceParams& P, const RowInfo& ri, int r, uint32_t off_lo,
                                             uint32_t off_hi)
{
    const int lane = threadIdx.x & 31;
    const int G = P.G;
    const SliceHdr* hd = P.hdr + size_t(r) * G;
    const SliceBody* bd = P.body + size_t(r) * G;
    K2 t{0ull, 0ull};
    uint32_t fl = 0;
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        const int b = lane + 32 * i;
        if (b < G) {
            fl |= __ldcg(&hd[b].flags);
            const uint4 g = __ldcg(reinterpret_cast<const uint4*>(&bd[b].ga));
            k2_insert(t, (static_cast<unsigned long long>(g.y) << 32) | g.x);
            k2_insert(t, (static_cast<unsigned long long>(g.w) << 32) | g.z);
        }
    }
    fl = warp_or(fl);
    k2_warp_reduce(t);
    const int32_t st = status_of(fl);
    int token = -1;
    if (!st) token = pick_of<InT>(P.k, ri, off_lo, off_hi, t);
    if (lane == 0) write_out(P.k, r, token, st);
}

// The digit d (0..255, bins[d] counts keys) where the count of keys in digits
// >= d first reaches `target`; `above` gets the count in digits > d. Lane L
// scans digits 255 - 8L down to 248 - 8L.
__device__ __forceinline__ int hist_pick(const uint32_t* bins, uint32_t target, uint32_t& above)
{
    const int lane = threadIdx.x & 31;
    uint32_t c[8], s = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        c[q] = bins[255 - (lane * 8 + q)];
        s += c[q];
    }
    uint32_t incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    uint32_t run = incl - s;
    int dig = -1;
    uint32_t abv = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        if (dig < 0 && run + c[q] >= target) {
            dig = 255 - (lane * 8 + q);
            abv = run;
        }
        run += c[q];
    }
    const uint32_t who = __ballot_sync(0xffffffffu, dig >= 0);
    const int src = who ? __ffs(who) - 1 : 0;
    above = __shfl_sync(0xffffffffu, abv, src);
    return who ? __shfl_sync(0xffffffffu, dig, src) : 0;
}

// A 16-bit prefix P with at least k of the row's sketch keys >= P << 16, and
// P << 16 at most the k-th largest of them (the row holds at least k keys).
// sk: the sketches of the row's slices, kSketch words each.
static __device__ __noinline__ uint32_t sketch_bound(const uint32_t* sk, int G, const uint32_t (&msk)[kSPL], int k,
                                                     uint32_t* bins)
{
    const int lane = threadIdx.x & 31;
    uint32_t pre = 0, target = uint32_t(k);
#pragma unroll 1
    for (int level = 0; level < 2; ++level) {
        for (int i = lane; i < 256; i += 32) bins[i] = 0;
        __syncwarp();
#pragma unroll 1
        for (int i = 0; i < kSPL; ++i) {
            const int b = lane + 32 * i;
            if (b >= G) break;
            for (uint32_t q = 0; q < msk[i]; ++q) {
                const uint32_t key = sk[b * kSketch + q];
                if (level == 1 && (key >> 24) != pre) continue;
                atomicAdd(&bins[level == 0 ? (key >> 24) : ((key >> 16) & 255u)], 1u);
            }
        }
        __syncwarp();
        uint32_t above;
        const int d = hist_pick(bins, target, above);
        __syncwarp();
        pre = level == 0 ? uint32_t(d) : (pre << 8) | uint32_t(d);
        target -= above;
    }
    return pre << 16;
}

// Keep, stably and at the front, the words whose key reaches lo; returns how
// many were kept.
__device__ __forceinline__ int compact_ge(unsigned long long* c, int n, uint32_t lo)
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

// The min-p threshold on the logit, m + T ln(min_p) in double precision,
// rounded up to fp32 (x >= result exactly when x >= the double threshold).
static __device__ __noinline__ float minp_threshold(float m, float T, float minp)
{
    const double th = double(m) + double(T) * log(double(minp));
    float t = float(th);
    if (double(t) < th) t = nextafterf(t, INFINITY);
    return t;
}

// The cuts over the sorted candidates of a truncated row, each keeping a prefix
// (top-k, then top-p over the top-k set or the whole row, then min-p), and the
// Gumbel pick over what is kept. Returns false when top-p reaches past the
// candidates of a row without top-k or min-p (the exact path takes it).
template <typename InT>
__device__ __forceinline__ bool cut_and_pick(const SliceParams& P, const RowInfo& ri, int r, uint32_t off_lo,
                                             uint32_t off_hi, const unsigned long long* cand, int C, float m,
                                             float xthr, const SliceHdr (&h)[kSPL], const SliceBody* bd, int G)
{
    const int lane = threadIdx.x & 31;
    const int nk = ri.do_topk ? ri.k : C;
    int nkeep = nk;
    if (ri.do_topp) {
        // fixed-point masses (2^-40 units of exp((x - m) / T)); keep while the
        // exclusive prefix mass is below p * Z
        double Zq;
        if (ri.do_topk) {
            unsigned long long s = 0;
            for (int i = lane; i < nk; i += 32) s += mass_q(key2f(cand_key(cand[i])), m, ri.invT);
            Zq = double(warp_sum_u64(s));
        } else {
            double z = 0.0;
#pragma unroll
            for (int i = 0; i < kSPL; ++i) {
                const int b = lane + 32 * i;
                if (b < G && h[i].mx > -INFINITY) {
                    const float zs = __ldcg(&bd[b].zs), zc = __ldcg(&bd[b].zc);
                    z += (double(zs) + double(zc)) * double(exp2f((h[i].mx - m) * ri.s2));
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
            Zq = z * 0x1p40;
        }
        const double target = double(ri.p) * Zq;
        unsigned long long base = 0;
        int cut = nk;
#pragma unroll 1
        for (int i0 = 0; i0 < nk; i0 += 32) {
            const int i = i0 + lane;
            const unsigned long long q = i < nk ? mass_q(key2f(cand_key(cand[i])), m, ri.invT) : 0ull;
            unsigned long long incl = q;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            const unsigned long long excl = base + incl - q;
            const uint32_t sb = __ballot_sync(0xffffffffu, i < nk && i > 0 && !(double(excl) < target));
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
        for (int i = lane; i < nkeep; i += 32) c += key2f(cand_key(cand[i])) >= xthr ? 1 : 0;
        nkeep = min(nkeep, int(__reduce_add_sync(0xffffffffu, uint32_t(c))));
    }
    nkeep = max(nkeep, 1);
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
    const int token = pick_of<InT>(P.k, ri, off_lo, off_hi, t);
    if (lane == 0) write_out(P.k, r, token, kRowOk);
    return true;
}

// Sort 32 * Q words held Q per lane (word q * 32 + lane), descending (bitonic).
template <int Q>
__device__ __forceinline__ void warp_sort_regs(unsigned long long (&a)[Q])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32 * Q; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 32) {
                const int qs = stride >> 5;
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    if ((q & qs) == 0) {
                        const int q2 = q | qs;
                        const bool desc = ((q * 32 + lane) & size) == 0;
                        const unsigned long long x = a[q], y = a[q2];
                        const bool sw = desc ? (x < y) : (x > y);
                        a[q] = sw ? y : x;
                        a[q2] = sw ? x : y;
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const bool desc = ((q * 32 + lane) & size) == 0;
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, a[q], stride);
                    const bool keep_max = desc == ((lane & stride) == 0);
                    a[q] = keep_max ? (a[q] > o ? a[q] : o) : (a[q] < o ? a[q] : o);
                }
            }
        }
    }
}

// Sort n words in warp-private shared memory, descending (bitonic through
// shared memory, padded with zeros up to a power of two; the buffer holds it).
static __device__ __noinline__ void warp_sort_smem(unsigned long long* a, int n)
{
    const int lane = threadIdx.x & 31;
    int np2 = 1;
    while (np2 < n) np2 <<= 1;
    for (int i = n + lane; i < np2; i += 32) a[i] = 0ull;
    __syncwarp();
#pragma unroll 1
    for (int size = 2; size <= np2; size <<= 1) {
#pragma unroll 1
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
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

// Sort the warp's n candidates, descending.
__device__ __forceinline__ void sort_cands(unsigned long long* c, int n)
{
    const int lane = threadIdx.x & 31;
    if (n <= 64) {
        unsigned long long a[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) a[q] = q * 32 + lane < n ? c[q * 32 + lane] : 0ull;
        warp_sort_regs<2>(a);
#pragma unroll
        for (int q = 0; q < 2; ++q) c[q * 32 + lane] = a[q];
        __syncwarp();
    } else {
        warp_sort_smem(c, n);
    }
}

__device__ __forceinline__ void cp_async_commit_wait()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Keep (at the front, in their order) the candidates whose key's top 16 bits
// reach those of the k-th largest key: the k largest words and their ties in
// that 16-bit bin. Returns how many were kept.
static __device__ __noinline__ int select_top(unsigned long long* c, int n, int k, uint32_t* bins)
{
    const int lane = threadIdx.x & 31;
    uint32_t pre = 0, target = uint32_t(k);
#pragma unroll 1
    for (int level = 0; level < 2; ++level) {
        for (int i = lane; i < 256; i += 32) bins[i] = 0;
        __syncwarp();
        for (int i = lane; i < n; i += 32) {
            const uint32_t key = cand_key(c[i]);
            if (level == 1 && (key >> 24) != pre) continue;
            atomicAdd(&bins[level == 0 ? (key >> 24) : ((key >> 16) & 255u)], 1u);
        }
        __syncwarp();
        uint32_t above;
        const int d = hist_pick(bins, target, above);
        __syncwarp();
        pre = level == 0 ? uint32_t(d) : (pre << 8) | uint32_t(d);
        target -= above;
    }
    return compact_ge(c, n, pre << 16);
}

// Append the finite tokens of slice b whose key reaches B to the candidates,
// reading the slice again from global memory.
template <typename InT>
__device__ __noinline__ void reread_slice(const SliceParams& P, const RowInfo& ri, int b, uint32_t B,
                                          unsigned long long* cand, int cap, uint32_t* count)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const int V = int(P.k.vocab);
    const int c0 = b * P.W;
    const int n = min(P.W, V - c0);
    SliceView<InT> sv;
    sv.sm = nullptr;
    sv.g = slice_ptr<InT>(P.k, ri.lrow, c0);
    sv.nb = 0;
    sv.nvec = (n + E - 1) / E;
    sv.n = n;
    sv.c0 = c0;
    const bool al = (reinterpret_cast<uintptr_t>(sv.g) & 15u) == 0;
    const uint4* gv = reinterpret_cast<const uint4*>(sv.g);
    for (int j = lane; j < sv.nvec; j += 32) {
        const uint4 v = (al && (j + 1) * E <= n) ? __ldg(gv + j) : sv.vec(j);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float x = Vec<InT>::get(v, e);
            if (x > -INFINITY && f2key(x) >= B) {
                const uint32_t pos = atomicAdd(count, 1u);
                if (pos < uint32_t(cap)) cand[pos] = cand_word(f2key(x), c0 + j * E + e);
            }
        }
    }
    __syncwarp();
}

// A truncated row from its slices' records. The warp's staging slot (idle at
// this point) is its scratch: the slices' sketches, then their lists, which
// become the candidates. All record loads go out in two rounds (headers and
// sketches, then the lists that matter). Returns false when the row must take
// the exact path (m out).
template <typename InT>
__device__ __forceinline__ bool finish_trunc(const SliceParams& P, WarpScratch& ws, const RowInfo& ri, int r,
                                             uint32_t off_lo, uint32_t off_hi, unsigned char* scratch, float& m_out)
{
    const int lane = threadIdx.x & 31;
    const int G = P.G;
    const SliceHdr* hd = P.hdr + size_t(r) * G;
    const SliceBody* bd = P.body + size_t(r) * G;
    uint32_t* sk = reinterpret_cast<uint32_t*>(scratch);  // [G][kSketch]
    unsigned long long* area = reinterpret_cast<unsigned long long*>(scratch + size_t(G) * kSketch * 4);
    const int cap = int((size_t(kSlotBytes) - size_t(G) * kSketch * 4) / 8);
    // round 1: headers and (tau, zs, zc, m) into registers, sketches into the scratch
    for (int b = lane; b < G; b += 32) {
        cp_async16(sk + b * kSketch, &bd[b].sketch[0]);
        cp_async16(sk + b * kSketch + 4, &bd[b].sketch[4]);
    }
    SliceHdr h[kSPL];
    uint32_t tau[kSPL], msk[kSPL];
    uint32_t fl = 0, nkeys = 0;
    float m = -INFINITY;
    int mi = INT_MAX;
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        const int b = lane + 32 * i;
        h[i].mx = -INFINITY;
        h[i].amax = INT_MAX;
        h[i].flags = 0;
        h[i].n = 0;
        tau[i] = 0;
        msk[i] = 0;
        if (b < G) {
            h[i] = ld_hdr(hd + b);
            const uint4 t4 = __ldcg(reinterpret_cast<const uint4*>(&bd[b].tau));
            tau[i] = t4.x;
            msk[i] = t4.w;
        }
    }
    cp_async_commit_wait();
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        fl |= h[i].flags;
        nkeys += msk[i];
        if (h[i].mx > m || (h[i].mx == m && h[i].amax < mi)) {
            m = h[i].mx;
            mi = h[i].amax;
        }
    }
    fl = warp_or(fl);
    nkeys = __reduce_add_sync(0xffffffffu, nkeys);
    warp_max_idx(m, mi);
    m_out = m;
    const int32_t st = status_of(fl);
    if (st) {
        if (lane == 0) write_out(P.k, r, -1, st);
        return true;
    }
    __syncwarp();
    // the min-p threshold on the logit: m + T ln(min_p), rounded up to fp32
    float xthr = -INFINITY;
    if (ri.do_minp) xthr = minp_threshold(m, ri.T, ri.minp);
    // B: every kept token's key reaches it
    uint32_t B;
    if (ri.do_topk) {
        if (ri.k > kKCap || nkeys < uint32_t(ri.k)) return false;
        B = sketch_bound(sk, G, msk, ri.k, ws.hist);
    } else if (ri.do_minp) {
        B = f2key(xthr);
    } else {
        uint32_t t = 0;
#pragma unroll
        for (int i = 0; i < kSPL; ++i) t = max(t, tau[i]);
        B = __reduce_max_sync(0xffffffffu, t);
    }
    B = max(B, 1u);
    // round 2: the lists of the slices that reach B and are complete above it,
    // copied side by side (even lengths; a padding entry is cleared); the
    // others are read again below
    uint32_t need = 0, mine = 0;
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        const int b = lane + 32 * i;
        if (b < G && h[i].mx != -INFINITY && f2key(h[i].mx) >= B) {
            if (h[i].n == kOverflow || tau[i] > B) need |= 2u << (2 * i);  // read again
            else {
                need |= 1u << (2 * i);
                mine += (h[i].n + 1u) & ~1u;
            }
        }
    }
    uint32_t incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    if (total > uint32_t(cap)) return false;
    uint32_t pos = incl - mine;
    uint32_t nre = 0;
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        const int b = lane + 32 * i;
        if (need & (1u << (2 * i))) {
            const uint32_t n2 = (h[i].n + 1u) & ~1u;
            for (uint32_t e = 0; e < n2; e += 2) cp_async16(area + pos + e, &bd[b].list[e]);
            pos += n2;
        }
        nre += (need >> (2 * i + 1)) & 1u;
    }
    cp_async_commit_wait();
    pos = incl - mine;
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        if (need & (1u << (2 * i))) {
            if (h[i].n & 1u) area[pos + h[i].n] = 0ull;
            pos += (h[i].n + 1u) & ~1u;
        }
    }
    __syncwarp();
    int C = compact_ge(area, int(total), B);
    // slices whose lists are not complete above B, read again
    if (__reduce_add_sync(0xffffffffu, nre) > uint32_t(kReCap)) return false;
    if (lane == 0) ws.n = uint32_t(C);
#pragma unroll 1
    for (int i = 0; i < kSPL; ++i) {
        const uint32_t who = __ballot_sync(0xffffffffu, (need >> (2 * i + 1)) & 1u);
        for (uint32_t w2 = who; w2; w2 &= w2 - 1) {
            __syncwarp();
            reread_slice<InT>(P, ri, (__ffs(w2) - 1) + 32 * i, B, area, cap, &ws.n);
        }
    }
    __syncwarp();
    C = int(ws.n);
    if (C > cap) return false;
    if (ri.do_topk && C < ri.k) return false;
    // top-k: bring the k largest to the front first when there are many more
    if (ri.do_topk && C > 64 && C > ri.k) C = select_top(area, C, ri.k, ws.hist);
    if (C > 64) {
        int np2 = 1;
        while (np2 < C) np2 <<= 1;
        if (np2 > cap) return false;
    }
    sort_cands(area, C);
    return cut_and_pick<InT>(P, ri, r, off_lo, off_hi, area, C, m, xthr, h, bd, G);
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

template <typename InT>
__device__ __forceinline__ float row_x(const KernelParams& kp, int lrow, int v)
{
    return ElemTraits<InT>::load(kp.logits, int64_t(lrow) * kp.row_stride + v);
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
            const float x = row_x<InT>(kp, ri.lrow, v);
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
            const float x = row_x<InT>(kp, ri.lrow, v);
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
__device__ __noinline__ void cta_exact_row(SliceShared& sh, const SliceParams& P, int r, const RowInfo& ri, float m,
                                           uint32_t off_lo, uint32_t off_hi)
{
    const KernelParams& kp = P.k;
    const int V = int(kp.vocab);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
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
    const RowPhilox rp = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, off_lo, off_hi);
    K2 t{0ull, 0ull};
    for (int v = tid; v < V; v += kT) {
        const float x = row_x<InT>(kp, ri.lrow, v);
        if (!(x > -INFINITY)) continue;
        if (hb && !in_prefix(f2key(x), v, bk, bi)) continue;
        if (ri.do_minp && !(x >= xthr)) continue;
        k2_insert(t, gkey(score2(x, ri.s2, philox_word(rp, v)), v));
    }
    k2_warp_reduce(t);
    if (lane == 0) {
        sh.red_k[2 * wid] = t.a;
        sh.red_k[2 * wid + 1] = t.b;
    }
    __syncthreads();
    if (wid == 0) {
        K2 a{0ull, 0ull};
        if (lane < kW) {
            a.a = sh.red_k[2 * lane];
            a.b = sh.red_k[2 * lane + 1];
        }
        k2_warp_reduce(a);
        const int token = pick_of<InT>(kp, ri, off_lo, off_hi, a);
        if (lane == 0) {
            write_out(kp, r, token, kRowOk);
            if (P.stats) atomicAdd(P.stats, 1ull);
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- one unit
// Wait for the warp's slot, summarise the unit into its record (row r, slice s).
template <typename InT>
__device__ __forceinline__ void process_unit(const SliceParams& P, const RowInfo& ri, uint64_t* bar,
                                             const unsigned char* slot, uint32_t parity, int r, int s,
                                             uint32_t off_lo, uint32_t off_hi)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const KernelParams& kp = P.k;
    const int G = P.G;
    uint32_t extra = 0;
    // when the wait gives up, the unit is marked and the copy is still awaited
    // (with a longer bound) before the slot is reused
    if (!mbar_wait_bounded(bar, parity, P.max_polls)) {
        extra = kFlagTimeout;
        mbar_wait_bounded(bar, parity, kDrainPolls);
    }
    if (ri.cls == kClsErr) return;
    const int c0 = s * P.W;
    const int n_el = min(P.W, int(kp.vocab) - c0);
    SliceView<InT> sv;
    sv.sm = reinterpret_cast<const uint4*>(slot);
    sv.g = slice_ptr<InT>(kp, ri.lrow, c0);
    sv.nb = bulk_vecs<InT>(sv.g, n_el);
    sv.nvec = (n_el + E - 1) / E;
    sv.n = n_el;
    sv.c0 = c0;
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
            int li;
            uint32_t f;
            lane_max<InT>(sv, lm, li, f);
            hdr.flags = warp_or(f);
            warp_max_idx(lm, li);
            hdr.mx = lm;
            hdr.amax = li;
        } else if (ri.cls == kClsPlain) {
            unit_plain<InT>(sv, ri, off_lo, off_hi, g, hdr.flags);
        } else {
            unit_trunc<InT>(sv, ri, hdr, body);
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
}

// Finish row r (this warp's arrival completed it); scratch: the warp's idle
// staging slot. Returns false when the row is left for the exact path.
template <typename InT>
__device__ __noinline__ bool finish_row(const SliceParams& P, WarpScratch& ws, const RowInfo& ri, int r,
                                        uint32_t off_lo, uint32_t off_hi, unsigned char* scratch, float& m)
{
    m = -INFINITY;
    if (ri.cls == kClsGreedy) {
        finish_greedy(P, r);
        return true;
    }
    if (ri.cls == kClsPlain) {
        finish_plain<InT>(P, ri, r, off_lo, off_hi);
        return true;
    }
    return finish_trunc<InT>(P, ws, ri, r, off_lo, off_hi, scratch, m);
}

// ---------------------------------------------------------------- the kernel
template <typename InT>
__global__ void __launch_bounds__(kT, 1) slice_kernel(const __grid_constant__ SliceParams P)
{
    extern __shared__ __align__(128) unsigned char smem[];
    SliceShared& sh = *reinterpret_cast<SliceShared*>(smem);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    unsigned char* slot = smem + kHead + size_t(wid) * kSlotBytes;
    uint64_t* bar = &sh.full[wid];
    WarpScratch& ws = sh.ws[wid];
    const KernelParams& kp = P.k;
    const int NC = int(gridDim.x);
    const int stride = NC * kW;
    int u = int(blockIdx.x) + wid * NC;  // round-robin over CTAs first
    // the copy of this warp's first unit goes out before anything else
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        if (u < P.n_units) issue_unit<InT>(P, bar, slot, u);
    }
    if (tid == 0) sh.n_exact = 0;
    const uint64_t off = kp.philox_offset_dev ? *kp.philox_offset_dev : kp.philox_offset;
    const uint32_t off_lo = uint32_t(off), off_hi = uint32_t(off >> 32);
    __syncthreads();  // n_exact is set before any warp can queue a row
    uint32_t parity = 0;
#pragma unroll 1
    while (u < P.n_units) {
        const int r = u / P.G, s = u - r * P.G;
        const RowInfo ri = load_info(P, r);
        process_unit<InT>(P, ri, bar, slot, parity, r, s, off_lo, off_hi);
        parity ^= 1u;
        const int un = u + stride;
        if (ri.cls == kClsErr) {
            if (s == 0 && lane == 0) write_out(kp, r, -1, kRowBadParam);
        } else {
            // the arrival is a release (publishing this unit's record) and an acquire
            // (seeing every other unit's record when it completes the row)
            __syncwarp();
            uint32_t old = 0;
            if (lane == 0) old = atom_add_acq_rel(&P.cnt[size_t(r) * kCntStride], 1u);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == uint32_t(P.G - 1)) {
                __syncwarp();
                float m;
                const bool done = finish_row<InT>(P, ws, ri, r, off_lo, off_hi, slot, m);
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
    // rows the candidate lists could not settle
    __syncthreads();
    const int ne = sh.n_exact;
    for (int q = 0; q < ne; ++q) {
        const int r = sh.exact_rows[q];
        cta_exact_row<InT>(sh, P, r, load_info(P, r), sh.exact_m[q], off_lo, off_hi);
    }
}

}  // namespace slc
}  // namespace dst
