// slice_kernel.cuh -- body of the slice kernel (design in slice_sampler.cuh).
//
// Every (row, slice) pays a fixed cost on top of its tokens, and there are
// rows x G of them, so the per-slice paths are written for few instructions:
// one exact score per lane seeds the plain-row bound, warp reductions work on
// 64-bit composite keys, each warp publishes all of its records behind one
// fence and one batch of atomics, and the double-precision settle of a pick
// runs only when the two best fp32 scores are within their error bound. Rare
// paths (list re-reads, large sorts, the exact path) stay out of line.
#pragma once

#include "slice_sampler.cuh"

namespace dst {
namespace slc {

// ---------------------------------------------------------------- set-up
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
    ri.m = uint8_t(ri.do_topk ? min(ri.k, kMLanes) : kMLanes);
    ri.aligned = 0;
    ri.pad = 0;
    if (bad) ri.cls = kClsErr;
    else if (greedy) ri.cls = kClsGreedy;
    else if (!ri.do_topk && !ri.do_topp && !ri.do_minp) ri.cls = kClsPlain;
    else ri.cls = kClsTrunc;
    return ri;
}

// First element of slice c0 of logits row lrow.
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

// Arm slot s for its next phase and start the copy of (lrow, this CTA's slice).
template <typename InT>
__device__ __forceinline__ void issue_copy(const SliceParams& P, SliceShared& sh, unsigned char* slots, int s,
                                           int lrow, int c0, int n)
{
    const InT* g = slice_ptr<InT>(P.k, lrow, c0);
    const int nb = bulk_vecs<InT>(g, n);
    const uint32_t bytes = uint32_t(nb) * 16u;
    mbar_arrive_expect_tx(&sh.full[s], bytes);
    if (bytes) bulk_copy_g2s(slots + size_t(s) * P.slot_bytes, g, bytes, &sh.full[s]);
}

// Atomic add with release and acquire semantics at GPU scope.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

template <typename InT>
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
// the slice a lane reads.
template <typename InT>
__device__ __forceinline__ void lane_max(const SliceView<InT>& sv, float& m, int& mi, uint32_t& f)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    m = -INFINITY;
    mi = INT_MAX;
    f = 0;
#pragma unroll 2
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

// ---------------------------------------------------------------- plain slice
// Every token of one vector whose score bound reaches thr is scored exactly
// into t (skipping the lane's seed token, already in t).
template <typename InT>
__device__ __forceinline__ void plain_vec(const uint4& v, int t0, const uint4& b0, const uint4& b1, float s2,
                                          float thr, int skip, K2& t)
{
    constexpr int E = Vec<InT>::E;
    uint32_t hit = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float x = Vec<InT>::get(v, e);
        const uint32_t we = lane_of(e < 4 ? b0 : b1, uint32_t(e) & 3u);
        // E >= 1 - u, so x/T - ln E <= x/T - ln(1 - u) (log2 units here)
        const float bound = fmaf(x, s2, -__log2f(noise_one_minus_u(we)));
        hit |= (bound >= thr ? 1u : 0u) << e;
    }
#pragma unroll 1
    for (; hit; hit &= hit - 1) {
        const int e = __ffs(hit) - 1;
        const int idx = t0 + e;
        const float x = Vec<InT>::get(v, e);
        if (idx == skip || !(x > -INFINITY)) continue;
        const uint32_t we = lane_of(e < 4 ? b0 : b1, uint32_t(e) & 3u);
        k2_insert(t, gkey(score2(x, s2, we), idx));
    }
}

template <typename InT>
__device__ __forceinline__ void slice_plain(const SliceView<InT>& sv, const RowInfo& ri, uint32_t off_lo,
                                            uint32_t off_hi, K2& out, uint32_t& flags)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    // each lane scores its largest logit exactly; the second-best of these 32
    // scores bounds the slice's second-best score from below
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
        const float ss = score2(lm, s2, philox_word<InT>(rp, li));
        t.a = gkey(ss, li);
        sk = f2key(ss);
    }
    uint32_t k1, k2;
    warp_top2_u32(sk, k1, k2);
    float thr = -INFINITY;
    if (k2 != 0) {
        thr = key2f(k2);
        thr -= 1e-4f + 4e-6f * fabsf(thr);
    }
    // every other token whose bound reaches thr, two vectors (up to four Philox
    // blocks) in flight per lane
    int j = lane;
#pragma unroll 1
    for (; j + 32 < sv.nvec; j += 64) {
        const int t0 = sv.c0 + j * E, t1 = t0 + 32 * E;
        const uint4 v0 = sv.vec(j), v1 = sv.vec(j + 32);
        const uint4 a0 = philox_block(rp, uint32_t(t0) >> 2);
        const uint4 c0 = philox_block(rp, uint32_t(t1) >> 2);
        uint4 a1 = a0, c1 = c0;
        if constexpr (E == 8) {
            a1 = philox_block(rp, (uint32_t(t0) >> 2) + 1u);
            c1 = philox_block(rp, (uint32_t(t1) >> 2) + 1u);
        }
        plain_vec<InT>(v0, t0, a0, a1, s2, thr, li, t);
        plain_vec<InT>(v1, t1, c0, c1, s2, thr, li, t);
    }
    if (j < sv.nvec) {
        const int t0 = sv.c0 + j * E;
        const uint4 v0 = sv.vec(j);
        const uint4 a0 = philox_block(rp, uint32_t(t0) >> 2);
        uint4 a1 = a0;
        if constexpr (E == 8) a1 = philox_block(rp, (uint32_t(t0) >> 2) + 1u);
        plain_vec<InT>(v0, t0, a0, a1, s2, thr, li, t);
    }
    k2_warp_reduce(t);
    out = t;
}

// ---------------------------------------------------------------- truncated slice
template <typename InT>
__device__ __forceinline__ void slice_trunc(const SliceView<InT>& sv, const RowInfo& ri, SliceHdr& hdr_out,
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
    // tau: the m-th largest lane maximum (as an order key); at least m tokens reach it
    const uint32_t lkey = lm > -INFINITY ? f2key(lm) : 0u;
    uint32_t left = lkey, tau = 0;
    for (int q = 0; q < int(ri.m); ++q) {
        tau = __reduce_max_sync(0xffffffffu, left);
        const uint32_t holder = __ballot_sync(0xffffffffu, left == tau);
        if (lane == __ffs(holder) - 1) left = 0;
    }
    tau = max(tau, 1u);  // -inf (key 0 here) is never listed
    // list every finite token whose key reaches tau: only lanes whose maximum
    // reaches it hold any
    uint32_t mine = 0;
    if (lkey >= tau) {
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
    // top-p rows without top-k: the slice's softmax mass at its maximum
    float zsum = 0.0f, zlow = 0.0f;
    if (ri.need_z && mx > -INFINITY && mx < INFINITY) {
        float zs = 0.0f, zc = 0.0f;  // Kahan: the sum is zs - zc
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
    if (lane == 0) {
        body->tau = tau;
        body->zs = zsum;
        body->zc = zlow;
    }
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

// The pick between the best two candidates in double precision (the oracle's
// definition); logits re-read, Philox words recomputed.
template <typename InT>
__device__ __noinline__ int settle_pair(const KernelParams& kp, const RowInfo& ri, uint32_t off_lo, uint32_t off_hi,
                                        unsigned long long a, unsigned long long b)
{
    const int ia = cand_idx(a), ib = cand_idx(b);
    const RowPhilox rp = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, off_lo, off_hi);
    const float xa = ElemTraits<InT>::load(kp.logits, int64_t(ri.lrow) * kp.row_stride + ia);
    const float xb = ElemTraits<InT>::load(kp.logits, int64_t(ri.lrow) * kp.row_stride + ib);
    const double sa = gumbel_score_f64(xa, ri.T, philox_word<InT>(rp, ia));
    const double sb = gumbel_score_f64(xb, ri.T, philox_word<InT>(rp, ib));
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

// Largest 16-bit key prefix P with at least k of the keys >= P << 16 (so
// P << 16 is at most the k-th largest key); missing keys are 0.
__device__ __forceinline__ uint32_t kth_lower_bound(const uint32_t (&key)[kSPL], int k)
{
    uint32_t pre = 0;
#pragma unroll 1
    for (int bit = 31; bit >= 16; --bit) {
        const uint32_t probe = pre | (1u << bit);
        uint32_t c = 0;
#pragma unroll
        for (int i = 0; i < kSPL; ++i) c += key[i] >= probe ? 1u : 0u;
        c = __reduce_add_sync(0xffffffffu, c);
        if (c >= uint32_t(k)) pre = probe;
    }
    return pre;
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

// Sort n <= kCandCap words in warp-private shared memory, descending (bitonic
// through shared memory, padded with zeros up to a power of two).
__device__ __noinline__ void warp_sort_smem(unsigned long long* a, int n)
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

// Sort the warp's n candidates (in its shared-memory buffer), descending.
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
    } else if (n <= 128) {
        unsigned long long a[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) a[q] = q * 32 + lane < n ? c[q * 32 + lane] : 0ull;
        warp_sort_regs<4>(a);
#pragma unroll
        for (int q = 0; q < 4; ++q) c[q * 32 + lane] = a[q];
        __syncwarp();
    } else {
        warp_sort_smem(c, n);
    }
}

// Append the finite tokens of slice b whose key reaches B to the warp's
// candidate buffer, reading the slice again from global memory.
template <typename InT>
__device__ __noinline__ void reread_slice(const SliceParams& P, SliceShared& sh, const RowInfo& ri, int b, uint32_t B)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
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
                const uint32_t pos = atomicAdd(&sh.wn[wid], 1u);
                if (pos < uint32_t(kCandCap)) sh.cand[wid][pos] = cand_word(f2key(x), c0 + j * E + e);
            }
        }
    }
    __syncwarp();
}

// A truncated row from its slices' records. Returns false when the row must
// take the exact path (m, amax out).
template <typename InT>
__device__ __forceinline__ bool finish_trunc(const SliceParams& P, SliceShared& sh, const RowInfo& ri, int r,
                                             uint32_t off_lo, uint32_t off_hi, float& m_out, int& amax_out)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int G = P.G;
    const SliceHdr* hd = P.hdr + size_t(r) * G;
    const SliceBody* bd = P.body + size_t(r) * G;
    SliceHdr h[kSPL];
    uint32_t tau[kSPL], mkey[kSPL];
    uint32_t fl = 0;
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
        if (b < G) {
            h[i] = ld_hdr(hd + b);
            tau[i] = __ldcg(&bd[b].tau);
        }
    }
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        mkey[i] = h[i].mx > -INFINITY ? f2key(h[i].mx) : 0u;
        fl |= h[i].flags;
        if (h[i].mx > m || (h[i].mx == m && h[i].amax < mi)) {
            m = h[i].mx;
            mi = h[i].amax;
        }
    }
    fl = warp_or(fl);
    warp_max_idx(m, mi);
    m_out = m;
    amax_out = mi;
    const int32_t st = status_of(fl);
    if (st) {
        if (lane == 0) write_out(P.k, r, -1, st);
        return true;
    }
    // the min-p threshold on the logit: m + T ln(min_p), rounded up to fp32
    float xthr = -INFINITY;
    if (ri.do_minp) {
        const double th = double(m) + double(ri.T) * log(double(ri.minp));
        float t = float(th);
        if (double(t) < th) t = nextafterf(t, INFINITY);
        xthr = t;
    }
    // B: every kept token's key reaches it
    uint32_t B;
    if (ri.do_topk) {
        if (ri.k > kKCap || G < ri.k) return false;
        B = kth_lower_bound(mkey, ri.k);
    } else if (ri.do_minp) {
        B = f2key(xthr);
    } else {
        uint32_t t = 0;
#pragma unroll
        for (int i = 0; i < kSPL; ++i) t = max(t, tau[i]);
        B = __reduce_max_sync(0xffffffffu, t);
    }
    B = max(B, 1u);
    // gather the listed tokens >= B; a slice whose list is not complete above B
    // is read again. All list loads of a lane are issued before any is used.
    if (lane == 0) {
        sh.wn[wid] = 0;
        sh.wre_n[wid] = 0;
    }
    __syncwarp();
    unsigned long long* cand = sh.cand[wid];
#pragma unroll
    for (int i = 0; i < kSPL; ++i) {
        const int b = lane + 32 * i;
        const bool need = b < G && mkey[i] >= B;
        const bool whole = need && h[i].n != kOverflow && tau[i] <= B;
        if (need && !whole) {
            const uint32_t q = atomicAdd(&sh.wre_n[wid], 1u);
            if (q < uint32_t(kReCap)) sh.wre[wid][q] = uint16_t(b);
        }
        const int n = whole ? int(h[i].n) : 0;
        unsigned long long w[kLCap];
#pragma unroll
        for (int e = 0; e < kLCap; e += 2) {
            if (e < n) {
                const ulonglong2 two = __ldcg(reinterpret_cast<const ulonglong2*>(&bd[b].list[e]));
                w[e] = two.x;
                w[e + 1] = two.y;
            } else {
                w[e] = 0ull;
                w[e + 1] = 0ull;
            }
        }
#pragma unroll
        for (int e = 0; e < kLCap; ++e) {
            if (e < n && cand_key(w[e]) >= B) {
                const uint32_t pos = atomicAdd(&sh.wn[wid], 1u);
                if (pos < uint32_t(kCandCap)) cand[pos] = w[e];
            }
        }
    }
    __syncwarp();
    const uint32_t nre = sh.wre_n[wid];
    if (nre > uint32_t(kReCap)) return false;
#pragma unroll 1
    for (uint32_t q = 0; q < nre; ++q) {
        reread_slice<InT>(P, sh, ri, sh.wre[wid][q], B);
        if (sh.wn[wid] > uint32_t(kCandCap)) break;
    }
    const int C = int(sh.wn[wid]);
    if (C > kCandCap) return false;
    sort_cands(cand, C);
    // the cuts, each keeping a prefix of the sorted candidates: top-k, then top-p
    // over the top-k set (or the whole row), then min-p
    int nk = C;
    if (ri.do_topk) {
        if (C < ri.k) return false;
        nk = ri.k;
    }
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
        if (!ri.do_topk && !ri.do_minp && cut == nk) return false;  // the cut lies past the lists
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
    for (int i = lane; i < nkeep; i += 32) {
        const unsigned long long c = cand[i];
        const int v = cand_idx(c);
        k2_insert(t, gkey(score2(key2f(cand_key(c)), ri.s2, philox_word<InT>(rp, v)), v));
    }
    k2_warp_reduce(t);
    const int token = pick_of<InT>(P.k, ri, off_lo, off_hi, t);
    if (lane == 0) write_out(P.k, r, token, kRowOk);
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
        k2_insert(t, gkey(score2(x, ri.s2, philox_word<InT>(rp, v)), v));
    }
    k2_warp_reduce(t);
    unsigned long long* red = reinterpret_cast<unsigned long long*>(sh.red_g);
    if (lane == 0) {
        red[2 * wid] = t.a;
        red[2 * wid + 1] = t.b;
    }
    __syncthreads();
    if (wid == 0) {
        K2 a{0ull, 0ull};
        if (lane < kW) {
            a.a = red[2 * lane];
            a.b = red[2 * lane + 1];
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

// ---------------------------------------------------------------- one (row, slice)
// Wait for the slot, summarise the slice into its record, free the slot for the
// next wave. The arrival on the row's counter comes later (batched per warp).
template <typename InT>
__device__ __forceinline__ void process_slice(const SliceParams& P, SliceShared& sh, unsigned char* slots, int r,
                                              int s, uint32_t parity, int c0, int n_el)
{
    constexpr int E = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const KernelParams& kp = P.k;
    const RowInfo ri = sh.info[r];
    const int N = P.n_rows, S = P.slots, G = P.G;
    uint32_t extra = 0;
    // when the wait gives up, the slice is marked and the copy is still awaited
    // (with a longer bound) before the slot is reused
    bool landed = mbar_wait_bounded(&sh.full[s], parity, P.max_polls);
    if (!landed) {
        extra = kFlagTimeout;
        landed = mbar_wait_bounded(&sh.full[s], parity, kDrainPolls);
    }
    SliceView<InT> sv;
    sv.sm = reinterpret_cast<const uint4*>(slots + size_t(s) * P.slot_bytes);
    sv.g = slice_ptr<InT>(kp, ri.lrow, c0);
    sv.nb = bulk_vecs<InT>(sv.g, n_el);
    sv.nvec = (n_el + E - 1) / E;
    sv.n = n_el;
    sv.c0 = c0;
    const uint32_t off_lo = sh.off_lo, off_hi = sh.off_hi;
    SliceHdr hdr;
    hdr.mx = -INFINITY;
    hdr.amax = INT_MAX;
    hdr.flags = kFlagAnyFinite;  // a slice that gave up reports only the timeout
    hdr.n = 0;
    K2 g{0ull, 0ull};
    SliceBody* body = P.body + size_t(r) * G + blockIdx.x;
    if (ri.cls != kClsErr && !extra) {
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
            slice_plain<InT>(sv, ri, off_lo, off_hi, g, hdr.flags);
        } else {
            slice_trunc<InT>(sv, ri, hdr, body);
        }
    }
    hdr.flags |= extra;
    // the slot is free: start the copy of the row this slot serves in the next wave
    __syncwarp();
    const int rn = r + S;
    if (lane == 0 && rn < N && landed) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_copy<InT>(P, sh, slots, s, sh.info[rn].lrow, c0, n_el);
    }
    if (ri.cls != kClsErr && lane == 0) {
        *reinterpret_cast<uint4*>(P.hdr + size_t(r) * G + blockIdx.x) =
            make_uint4(__float_as_uint(hdr.mx), uint32_t(hdr.amax), hdr.flags, hdr.n);
        if (ri.cls == kClsPlain)
            *reinterpret_cast<uint4*>(&body->ga) =
                make_uint4(uint32_t(g.a), uint32_t(g.a >> 32), uint32_t(g.b), uint32_t(g.b >> 32));
    }
}

// Finish row r (this warp's arrival completed it).
template <typename InT>
__device__ __noinline__ void finish_row(const SliceParams& P, SliceShared& sh, int r)
{
    const int lane = threadIdx.x & 31;
    const RowInfo ri = sh.info[r];
    const uint32_t off_lo = sh.off_lo, off_hi = sh.off_hi;
    if (ri.cls == kClsGreedy) {
        finish_greedy(P, r);
    } else if (ri.cls == kClsPlain) {
        finish_plain<InT>(P, ri, r, off_lo, off_hi);
    } else {
        float m;
        int amax;
        if (!finish_trunc<InT>(P, sh, ri, r, off_lo, off_hi, m, amax) && lane == 0) {
            const int q = atomicAdd(&sh.n_exact, 1);
            sh.exact_rows[q] = r;
            sh.exact_m[q] = m;
            sh.exact_amax[q] = amax;
        }
    }
    if (lane == 0) P.cnt[size_t(r) * kCntStride] = 0;
}

// ---------------------------------------------------------------- the kernel
template <typename InT>
__global__ void __launch_bounds__(kT, 1) slice_kernel(const __grid_constant__ SliceParams P)
{
    extern __shared__ __align__(128) unsigned char smem[];
    SliceShared& sh = *reinterpret_cast<SliceShared*>(smem);
    unsigned char* slots = smem + kHead;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int N = P.n_rows, S = P.slots, G = P.G;
    const int c0 = int(blockIdx.x) * P.W;
    const int n_el = min(P.W, int(P.k.vocab - c0));
    const int nfirst = min(S, N);
    const KernelParams& kp = P.k;
    constexpr int kCopyWarp = kW - 1;  // issues the copies while other warps read parameters

    if (tid == 0) {
        for (int s = 0; s < nfirst; ++s) mbar_init(&sh.full[s], 1);
        fence_mbar_init();
        sh.n_exact = 0;
    }
    __syncthreads();
    const bool direct = kp.logit_row == nullptr;
    if (direct && wid == kCopyWarp)
        for (int s = lane; s < nfirst; s += 32) issue_copy<InT>(P, sh, slots, s, s, c0, n_el);
    if (tid < N) sh.info[tid] = load_info(P, tid);
    if (tid == kT - 1) {
        const uint64_t off = kp.philox_offset_dev ? *kp.philox_offset_dev : kp.philox_offset;
        sh.off_lo = uint32_t(off);
        sh.off_hi = uint32_t(off >> 32);
    }
    __syncthreads();
    if (!direct && wid == kCopyWarp)
        for (int s = lane; s < nfirst; s += 32) issue_copy<InT>(P, sh, slots, s, sh.info[s].lrow, c0, n_el);
    // order each wave's rows by kind: truncated, plain, greedy, bad parameter
    // (waves are runs of S rows; S is a multiple of 32 whenever there are several,
    // so a group of 32 rows never spans two waves)
    {
        const int r = tid;
        const int c = r < N ? int(sh.info[r].cls) : 4;
        uint32_t bal[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) bal[q] = __ballot_sync(0xffffffffu, c == q);
        if (lane == 0 && wid < kMaxRows / 32)
#pragma unroll
            for (int q = 0; q < 4; ++q) sh.wcls[wid][q] = __popc(bal[q]);
        __syncthreads();
        if (r < N) {
            const int w0 = (r / S) * S, wend = min(N, w0 + S);
            int pos = w0;
            for (int q = 0; q < c; ++q)
                for (int g32 = w0 >> 5; g32 < ((wend + 31) >> 5); ++g32) pos += int(sh.wcls[g32][q]);
            for (int g32 = w0 >> 5; g32 < (r >> 5); ++g32) pos += int(sh.wcls[g32][c]);
            pos += __popc(bal[c] & ((1u << lane) - 1u));
            sh.order[pos] = uint16_t(r);
        }
        __syncthreads();
    }
    // bad-parameter rows are answered once, by CTA 0
    if (blockIdx.x == 0 && tid < N && sh.info[tid].cls == kClsErr) write_out(kp, tid, -1, kRowBadParam);
    // the waves. A slot's wait on the parity of wave w + 1 must not start before
    // its wave-w phase has completed (a parity wait two phases ahead returns at
    // once), so the CTA meets at a barrier between waves; by then every slot of
    // wave w has been consumed and refilled.
    for (int w0 = 0; w0 < N; w0 += S) {
        const int wn = min(S, N - w0);
        const uint32_t parity = uint32_t(w0 / S) & 1u;
        int nmine = 0;
        for (int i = wid; i < wn; i += kW) {
            const int r = sh.order[w0 + i];
            process_slice<InT>(P, sh, slots, r, r - w0, parity, c0, n_el);
            if (sh.info[r].cls != kClsErr) {
                if (lane == 0) sh.wrow[wid][nmine] = uint16_t(r);
                ++nmine;
            }
        }
        // arrive on every row this warp sampled at once. The warp barrier orders
        // all lanes' record stores before the arrivals, and each arrival is a
        // release (publishing them) and an acquire (seeing every other slice's
        // records when it completes the row); then finish the completed rows
        __syncwarp();
        uint32_t last = 0;
        if (lane < nmine) {
            const int r = sh.wrow[wid][lane];
            last = atom_add_acq_rel(&P.cnt[size_t(r) * kCntStride], 1u) == uint32_t(G - 1) ? 1u : 0u;
        }
        uint32_t lmask = __ballot_sync(0xffffffffu, last != 0);
        if (lmask) __syncwarp();  // the other lanes read after the acquiring lane
        for (; lmask; lmask &= lmask - 1) finish_row<InT>(P, sh, sh.wrow[wid][__ffs(lmask) - 1]);
        if (w0 + S < N) __syncthreads();
    }
    // rows the candidate lists could not settle
    __syncthreads();
    const int ne = sh.n_exact;
    for (int q = 0; q < ne; ++q)
        cta_exact_row<InT>(sh, P, sh.exact_rows[q], sh.info[sh.exact_rows[q]], sh.exact_m[q], sh.off_lo, sh.off_hi);
}

}  // namespace slc
}  // namespace dst
