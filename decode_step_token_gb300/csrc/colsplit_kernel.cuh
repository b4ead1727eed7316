// colsplit_kernel.cuh -- body of the unit-split kernel (design in colsplit.cuh).
//
// Per warp and unit: the unit's logits go to the warp's shared-memory slot by
// 16-byte cp.async copies in kStages commit groups, the row's parameters are
// read while they fly, and the class pass (greedy / plain / truncated) starts on
// the first group as soon as it has landed. Loops over a unit's vectors stay
// rolled, and every pass, the finisher and the exact path are out-of-line, which
// keeps the code each warp runs small.
#pragma once

#include <cuda_bf16.h>

#include "colsplit.cuh"

namespace dst {
namespace col {

static_assert(kStages == 4, "wait_stage below spells out four stages");

__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t* p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Wait until copy group `st` of this warp has landed and is visible to all lanes.
__device__ __forceinline__ void wait_stage(int st)
{
    if (st == 0) cp_async_wait<3>();
    else if (st == 1) cp_async_wait<2>();
    else if (st == 2) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncwarp();
}

// One warp's unit: row r, elements [v0, v0 + n) staged as nvec 16-byte vectors,
// q vectors per copy group.
struct Unit {
    int r, s, v0, n, nvec, q;
};

// ---------------------------------------------------------------- row parameters
// Every lane reads the same words (one request each), all independent, so they
// share one memory round trip.
__device__ __forceinline__ RowInfo load_row_info(const ColParams& P, int r, int lrow)
{
    const KernelParams& kp = P.k;
    const int64_t V = kp.vocab;
    RowInfo ri;
    ri.T = kp.temperature[r];
    ri.k = kp.top_k ? kp.top_k[r] : -1;
    ri.p = kp.top_p ? kp.top_p[r] : 1.0f;
    ri.minp = kp.min_p ? kp.min_p[r] : 0.0f;
    const float pres = kp.presence ? kp.presence[r] : 0.0f;
    const float freq = kp.frequency ? kp.frequency[r] : 0.0f;
    const float rep = kp.repetition ? kp.repetition[r] : 1.0f;
    const bool seeded = kp.has_seed ? kp.has_seed[r] != 0 : false;
    const uint64_t row_seed = kp.seed ? kp.seed[r] : 0ull;
    const uint32_t row_stream = kp.stream_id ? kp.stream_id[r] : 0u;
    const uint64_t off = kp.philox_offset_dev ? *kp.philox_offset_dev : kp.philox_offset;
    const uint64_t key = seeded ? row_seed : kp.global_seed;
    const uint32_t sid = kp.stream_id ? row_stream : (seeded ? 0u : uint32_t(r));
    ri.stream = (sid & 0x7FFFFFFFu) | (seeded ? 0x80000000u : 0u);
    ri.key_lo = uint32_t(key);
    ri.key_hi = uint32_t(key >> 32);
    ri.off_lo = uint32_t(off);
    ri.off_hi = uint32_t(off >> 32);
    ri.lrow = lrow < 0 ? 0 : lrow;
    bool bad = lrow < 0;
    if (!(ri.T >= 0.0f) || isinf(ri.T)) bad = true;
    if (!(ri.k == -1 || ri.k >= 1)) bad = true;
    if (!(ri.p > 0.0f && ri.p <= 1.0f)) bad = true;
    if (!(ri.minp >= 0.0f && ri.minp <= 1.0f)) bad = true;
    if (!isfinite(pres) || !isfinite(freq)) bad = true;
    if (!(rep > 0.0f) || isinf(rep)) bad = true;
    ri.status = bad ? kRowBadParam : kRowOk;
    ri.greedy = ri.T < 1e-5f;
    ri.Te = ri.greedy ? 1.0f : ri.T;
    ri.invT = 1.0f / ri.Te;
    ri.do_topk = (ri.k != -1 && int64_t(ri.k) < V);
    ri.do_topp = ri.p < 1.0f;
    ri.do_minp = ri.minp > 0.0f;
    ri.small_k = ri.do_topk && ri.k <= kKeepCap;
    ri.need_z = ri.do_topp && !ri.do_topk;
    if (bad) ri.cls = kClsErr;
    else if (ri.greedy) ri.cls = kClsGreedy;
    else if (!ri.do_topk && !ri.do_topp && !ri.do_minp) ri.cls = kClsPlain;
    else ri.cls = kClsCand;
    return ri;
}

// ---------------------------------------------------------------- staging a unit
// Issue the unit's copies (kStages groups, always committed so that the waits
// line up), then build the vectors that cannot be copied whole -- the ragged
// last one, or all of them when the row start is not 16-byte aligned -- from
// plain loads, padded with -inf.
template <typename InT>
__device__ __forceinline__ void stage_unit(const KernelParams& kp, int lrow, Unit& u, uint4* slot)
{
    constexpr int ES = int(sizeof(InT));
    constexpr int EPV = 16 / ES;
    const int lane = threadIdx.x & 31;
    const int n = u.n;
    u.nvec = (n + EPV - 1) / EPV;
    u.q = ((u.nvec + kStages - 1) / kStages + 31) & ~31;
    const unsigned char* g = static_cast<const unsigned char*>(kp.logits) +
                             (int64_t(lrow < 0 ? 0 : lrow) * kp.row_stride + u.v0) * ES;
    const bool aligned = (reinterpret_cast<uintptr_t>(g) & 15u) == 0;
    const int nfull = (n > 0 && aligned) ? n / EPV : 0;
#pragma unroll 1
    for (int st = 0; st < kStages; ++st) {
        const int e = min((st + 1) * u.q, nfull);
        for (int j = st * u.q + lane; j < e; j += 32) cp_async16(slot + j, g + 16 * size_t(j));
        cp_async_commit();
    }
#pragma unroll 1
    for (int j = nfull + lane; j < u.nvec; j += 32) {
        uint32_t e[4];
#pragma unroll
        for (int q = 0; q < EPV; ++q) {
            const int i = j * EPV + q;
            if (ES == 2) {
                uint32_t b = 0xFF80u;  // bf16 -inf
                if (i < n) b = reinterpret_cast<const uint16_t*>(g)[i];
                if (q & 1) e[q >> 1] |= b << 16;
                else e[q >> 1] = b;
            } else {
                uint32_t b = 0xFF800000u;  // fp32 -inf
                if (i < n) b = reinterpret_cast<const uint32_t*>(g)[i];
                e[q] = b;
            }
        }
        slot[j] = make_uint4(e[0], e[1], e[2], e[3]);
    }
}

// ---------------------------------------------------------------- vector helpers
// The 8 (bf16) or 4 (fp32) logits of a 16-byte vector.
template <typename InT>
struct Vec;

template <>
struct Vec<uint16_t> {
    static constexpr int E = 8;
    // maximum of the vector (NaN ignored) and whether it holds a NaN
    __device__ static __forceinline__ float vmax(const uint4& r, bool& nan)
    {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
        const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
        const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));          // NaN ignored
        const __nv_bfloat162 mn = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));  // NaN kept
        const float n0 = __low2float(mn), n1 = __high2float(mn);
        nan = (n0 != n0) || (n1 != n1);
        return fmaxf(__low2float(m), __high2float(m));
    }
    __device__ static __forceinline__ float get(const uint4& r, int e) { return ElemTraits<uint16_t>::get(r, e); }
};

template <>
struct Vec<float> {
    static constexpr int E = 4;
    __device__ static __forceinline__ float vmax(const uint4& r, bool& nan)
    {
        const float a = __uint_as_float(r.x), b = __uint_as_float(r.y);
        const float c = __uint_as_float(r.z), d = __uint_as_float(r.w);
        nan = (a != a) || (b != b) || (c != c) || (d != d);
        return fmaxf(fmaxf(a, b), fmaxf(c, d));
    }
    __device__ static __forceinline__ float get(const uint4& r, int e) { return ElemTraits<float>::get(r, e); }
};

// First position of value m in the vector (m is one of its elements).
template <typename InT>
__device__ __forceinline__ int vec_find(const uint4& r, float m)
{
    int pos = Vec<InT>::E - 1;
#pragma unroll
    for (int e = Vec<InT>::E - 1; e >= 0; --e)
        if (Vec<InT>::get(r, e) == m) pos = e;
    return pos;
}

__device__ __forceinline__ uint32_t unit_flags(float lane_max, bool lane_nan)
{
    const bool bad = __any_sync(0xffffffffu, lane_nan || lane_max > 3.402823466e38f);
    const bool fin = __any_sync(0xffffffffu, lane_max > -INFINITY && !(lane_max > 3.402823466e38f));
    return (bad ? kFlagNonFinite : 0u) | (fin ? kFlagAnyFinite : 0u);
}

__device__ __forceinline__ void warp_maxidx(float& m, int& i)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, off);
        const int oi = __shfl_xor_sync(0xffffffffu, i, off);
        maxidx_merge(m, i, om, oi);
    }
}

// ---------------------------------------------------------------- greedy units
template <typename InT>
__device__ __noinline__ void unit_greedy(const Unit u, const uint4* slot, ColRec* rec)
{
    constexpr int EPV = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    float mx = -INFINITY;
    int am = INT_MAX;
    bool nan = false;
#pragma unroll 1
    for (int st = 0; st < kStages; ++st) {
        wait_stage(st);
        const int e = min((st + 1) * u.q, u.nvec);
#pragma unroll 1
        for (int j = st * u.q + lane; j < e; j += 32) {
            const uint4 raw = slot[j];
            bool vn;
            const float m = Vec<InT>::vmax(raw, vn);
            nan |= vn;
            if (m > mx) {
                mx = m;
                am = u.v0 + j * EPV + vec_find<InT>(raw, m);
            }
        }
    }
    const uint32_t flags = unit_flags(mx, nan);
    warp_maxidx(mx, am);
    if (lane == 0) {
        rec->mx = mx;
        rec->amax = am;
        rec->flags = flags;
        rec->nc = 0;
    }
}

// ---------------------------------------------------------------- plain temperature units
__device__ __forceinline__ float fast_ln_exp1(float w, float lg2w, uint32_t word)
{
    // small w: -ln(1 - w) = w (1 + w/2 + w^2/3 + ...), so ln E = ln w + w/2 + 5w^2/24 + w^3/8
    const float series = fmaf(lg2w, 0.69314718055994531f, w * fmaf(w, fmaf(w, 0.125f, 0.20833333f), 0.5f));
    const float direct = __logf(-__logf(noise_u(word)));
    return w < 0.03125f ? series : direct;
}

struct PlainAcc {
    GRec best;  // this lane's best token so far (fp32 score)
    float c2;   // entry bar in the log2 domain: -(best - margin) * log2 e
};

__device__ __forceinline__ float bar_of(float s)
{
    return -(s - (1e-4f + 1e-6f * fabsf(s))) * 1.4426950408889634f;
}

__device__ __forceinline__ void plain_take(PlainAcc& a, float invT, int v, float x, uint32_t word)
{
    const float w = noise_one_minus_u(word);
    const float s = x * invT - fast_ln_exp1(w, __log2f(w), word);
    if (s > a.best.s || (s == a.best.s && v < a.best.idx)) {
        a.best = GRec{s, v, x, word};
        a.c2 = bar_of(s);
    }
}

template <int E>
__device__ __forceinline__ float pickf(const float (&a)[E], int e)
{
    float r = a[0];
#pragma unroll
    for (int i = 1; i < E; ++i) r = (e == i) ? a[i] : r;
    return r;
}

template <int E>
__device__ __forceinline__ uint32_t picku(const uint32_t (&a)[E], int e)
{
    uint32_t r = a[0];
#pragma unroll
    for (int i = 1; i < E; ++i) r = (e == i) ? a[i] : r;
    return r;
}

// Gumbel-max over the unit: a token may win only if x/T - ln(1 - u) clears the
// lane's bar (its best score so far, less a margin); the exact score is taken
// only for those.
template <typename InT>
__device__ __noinline__ void unit_plain(const Unit u, const RowInfo ri, const uint4* slot, ColRec* rec)
{
    constexpr int EPV = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const float invT = ri.invT;
    const float a2 = invT * 1.4426950408889634f;
    const PhiloxKey key{ri.key_lo, ri.key_hi};
    const uint32_t stream = ri.stream, olo = ri.off_lo, ohi = ri.off_hi;
    PlainAcc a;
    a.best = grec_empty();
    a.c2 = INFINITY;
    float lm = -INFINITY;
    bool nan = false;
#pragma unroll 1
    for (int st = 0; st < kStages; ++st) {
        wait_stage(st);
        const int e = min((st + 1) * u.q, u.nvec);
#pragma unroll 1
        for (int j = st * u.q + lane; j < e; j += 32) {
            const int vb = u.v0 + j * EPV;  // a multiple of 4
            const uint4 raw = slot[j];
            bool vn;
            lm = fmaxf(lm, Vec<InT>::vmax(raw, vn));
            nan |= vn;
            float xs[EPV];
            uint32_t ws[EPV];
#pragma unroll
            for (int b = 0; b < EPV / 4; ++b) {
                const uint4 blk = philox4x32_10(make_uint4(uint32_t(vb >> 2) + b, stream, olo, ohi), key);
                ws[4 * b + 0] = blk.x;
                ws[4 * b + 1] = blk.y;
                ws[4 * b + 2] = blk.z;
                ws[4 * b + 3] = blk.w;
            }
            uint32_t mask = 0;
#pragma unroll
            for (int q = 0; q < EPV; ++q) {
                xs[q] = Vec<InT>::get(raw, q);
                const float lg2w = __log2f(noise_one_minus_u(ws[q]));
                mask |= (fmaf(xs[q], a2, a.c2) > lg2w) ? (1u << q) : 0u;
            }
            while (mask) {
                const int q = __ffs(mask) - 1;
                mask &= mask - 1;
                plain_take(a, invT, vb + q, pickf<EPV>(xs, q), picku<EPV>(ws, q));
            }
        }
    }
    const uint32_t flags = unit_flags(lm, nan);
    GTop2 t;
    t.a = a.best;
    t.b = grec_empty();
    top2_warp_reduce(t);
    if (lane == 0) {
        rec->mx = 0.0f;
        rec->amax = 0;
        rec->flags = flags;
        rec->nc = 0;
        rec->g0 = t.a;
        rec->g1 = t.b;
    }
}

// ---------------------------------------------------------------- word sorts
// Sort buf[0, n) descending, n <= kBufCap: in registers up to 128 words.
__device__ __noinline__ void sort_buf(unsigned long long* buf, int n)
{
    const int lane = threadIdx.x & 31;
    if (n <= 1) return;
    if (n <= 64) {
        unsigned long long a[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) a[q] = q * 32 + lane < n ? buf[q * 32 + lane] : 0ull;
        __syncwarp();
        warp_sort_regs_desc<2>(a);
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (q * 32 + lane < n) buf[q * 32 + lane] = a[q];
    } else if (n <= 128) {
        unsigned long long a[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) a[q] = q * 32 + lane < n ? buf[q * 32 + lane] : 0ull;
        __syncwarp();
        warp_sort_regs_desc<4>(a);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q * 32 + lane < n) buf[q * 32 + lane] = a[q];
    } else {
        warp_sort_smem_desc(buf, n);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- truncated units
// The unit's top-C list (C = k for k <= 64, else 64) by (value desc, index asc):
// every element at or above tau, the C-th largest of 64 group maxima (each lane
// keeps one maximum for its even and one for its odd vectors), is gathered and
// sorted. At least C elements reach tau, so the list is exact.
template <typename InT>
__device__ __noinline__ void unit_cand(const Unit u, const RowInfo ri, const uint4* slot,
                                       unsigned long long* buf, ColRec* rec)
{
    constexpr int EPV = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const int C = ri.small_k ? ri.k : kCandCap;
    float mx = -INFINITY, gm0 = -INFINITY, gm1 = -INFINITY;
    int am = INT_MAX;
    bool nan = false;
#pragma unroll 1
    for (int st = 0; st < kStages; ++st) {
        wait_stage(st);
        const int e = min((st + 1) * u.q, u.nvec);
#pragma unroll 1
        for (int j = st * u.q + lane; j < e; j += 32) {
            const uint4 raw = slot[j];
            bool vn;
            const float m = Vec<InT>::vmax(raw, vn);
            nan |= vn;
            if (m > mx) {
                mx = m;
                am = u.v0 + j * EPV + vec_find<InT>(raw, m);
            }
            if ((j >> 5) & 1) gm1 = fmaxf(gm1, m);
            else gm0 = fmaxf(gm0, m);
        }
    }
    const uint32_t flags = unit_flags(mx, nan);
    warp_maxidx(mx, am);
    const uint32_t gk[2] = {f2key(gm0), f2key(gm1)};
    const float tau = key2f(warp_kth_key<2>(gk, 3u, C));
    // gather x >= tau (finite) and, for top-p without top-k, the unit's softmax mass
    int cnt = 0;
    float zs = 0.0f, zc = 0.0f;
    const bool need_z = ri.need_z;
    const float invT = ri.invT;
#pragma unroll 1
    for (int j0 = 0; j0 < u.nvec; j0 += 32) {
        const int j = j0 + lane;
        const bool in = j < u.nvec;
        const uint4 raw = in ? slot[j] : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        const int vb = u.v0 + j * EPV;
        uint32_t mask = 0;
#pragma unroll
        for (int q = 0; q < EPV; ++q) {
            const float x = in ? Vec<InT>::get(raw, q) : -INFINITY;
            mask |= (x >= tau && x > -INFINITY) ? (1u << q) : 0u;
            if (need_z && x > -INFINITY) {
                const float y = __expf((x - mx) * invT) - zc;
                const float s2 = zs + y;
                zc = (s2 - zs) - y;
                zs = s2;
            }
        }
        if (__any_sync(0xffffffffu, mask != 0)) {
#pragma unroll
            for (int q = 0; q < EPV; ++q) {
                const bool take = (mask >> q) & 1u;
                const unsigned bt = __ballot_sync(0xffffffffu, take);
                if (take) {
                    const int pos = cnt + __popc(bt & ((1u << lane) - 1u));
                    if (pos < kBufCap) buf[pos] = comp_of(Vec<InT>::get(raw, q), vb + q);
                }
                cnt += __popc(bt);
            }
        }
    }
    __syncwarp();
    if (need_z) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, zs, off);
            const float oc = __shfl_xor_sync(0xffffffffu, zc, off);
            const float y = os - oc - zc;
            const float s2 = zs + y;
            zc = (s2 - zs) - y;
            zs = s2;
        }
    }
    uint32_t nc;
    if (cnt > kBufCap) {
        nc = kOverflow;
    } else {
        sort_buf(buf, cnt);
        nc = uint32_t(min(cnt, C));
        for (int i = lane; i < int(nc); i += 32) rec->cand[i] = buf[i];
    }
    if (lane == 0) {
        rec->mx = mx;
        rec->amax = am;
        rec->flags = flags;
        rec->nc = nc;
        rec->zs = zs;
        rec->zc = zc;
    }
}

// ---------------------------------------------------------------- finishing a row
__device__ __noinline__ int settle_slow(const GTop2 t, float T) { return settle_top2(t, T); }

// Pick between the two best fp32 Gumbel candidates; double precision only when
// they are within fp32 reach of each other.
__device__ __forceinline__ int settle_fast(const GTop2& t, float T)
{
    if (t.a.idx == INT_MAX) return -1;
    if (t.b.idx == INT_MAX) return t.a.idx;
    const float tol = 1e-4f + 1e-5f * fmaxf(fabsf(t.a.s), fabsf(t.b.s));
    if (t.a.s - t.b.s > tol) return t.a.idx;
    return settle_slow(t, T);
}

// Fast fp32 Gumbel record of a kept candidate.
__device__ __forceinline__ GRec cand_grec(const RowInfo& ri, float x, int v)
{
    const uint4 blk = philox4x32_10(make_uint4(uint32_t(v) >> 2, ri.stream, ri.off_lo, ri.off_hi),
                                    PhiloxKey{ri.key_lo, ri.key_hi});
    const uint32_t word = lane_of(blk, uint32_t(v) & 3u);
    const float w = noise_one_minus_u(word);
    return GRec{x * ri.invT - fast_ln_exp1(w, __log2f(w), word), v, x, word};
}

// Append to buf[n, ...) every listed word whose value key is >= vt, reading
// each list from its head 8 words at a time and leaving it at its first word
// below vt; returns the new count (only the first kBufCap words are stored).
__device__ __forceinline__ int gather_lists(const ColRec* rr, int G, const uint32_t (&nc)[kLPL], uint32_t vt,
                                            unsigned long long* buf, int n)
{
    const int lane = threadIdx.x & 31;
    int len[kLPL];
#pragma unroll
    for (int q = 0; q < kLPL; ++q) len[q] = int(nc[q]);
#pragma unroll 1
    for (int i0 = 0; i0 < kCandCap; i0 += 8) {
        bool more = false;
#pragma unroll
        for (int q = 0; q < kLPL; ++q) more |= i0 < len[q];
        if (!__any_sync(0xffffffffu, more)) break;
        unsigned long long w[kLPL][8];
#pragma unroll
        for (int q = 0; q < kLPL; ++q) {
            const int s = lane + 32 * q;
            if (i0 < len[q]) {
                const uint4* src = reinterpret_cast<const uint4*>(&rr[s].cand[i0]);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint4 x = __ldcg(src + h);
                    w[q][2 * h] = (static_cast<unsigned long long>(x.y) << 32) | x.x;
                    w[q][2 * h + 1] = (static_cast<unsigned long long>(x.w) << 32) | x.z;
                }
            } else {
#pragma unroll
                for (int h = 0; h < 8; ++h) w[q][h] = 0ull;
            }
        }
#pragma unroll
        for (int q = 0; q < kLPL; ++q) {
            if (!__any_sync(0xffffffffu, i0 < len[q])) continue;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const bool take = i0 + h < len[q] && cand_key(w[q][h]) >= vt;
                const unsigned bt = __ballot_sync(0xffffffffu, take);
                if (take) {
                    const int pos = n + __popc(bt & ((1u << lane) - 1u));
                    if (pos < kBufCap) buf[pos] = w[q][h];
                }
                n += __popc(bt);
            }
            if (!(cand_key(w[q][7]) >= vt)) len[q] = 0;  // sorted: the rest is below vt
        }
    }
    __syncwarp();
    return n;
}

// The kept set of a truncated row from its units' lists; returns the token, or
// sets `fallback` when the lists cannot settle it. hd: the headers of the
// lane's lists (list lane + 32 q).
__device__ __noinline__ int finish_cand(const ColParams& P, unsigned long long* buf, const RowInfo ri,
                                        const ColRec* rr, const uint32_t (&nc)[kLPL], float m, bool& fallback)
{
    const int lane = threadIdx.x & 31;
    const int G = P.gc;
    const bool small_k = ri.small_k;
    const int C = small_k ? ri.k : kCandCap;
    int token = -1;
    if (ri.do_topk && !small_k) {
        fallback = true;
        return -1;
    }
    // one round trip: the C-th word of every list, and a sample of h words from
    // the head of every list (G h >= C of them when the lists hold that many)
    const int h = min(C, (C + G - 1) / G);
    const int ns = G * h;  // <= G + C - 1 <= 191
    constexpr int kSPL = 6;
    unsigned long long tail[kLPL];
    uint32_t sk[kSPL];
    uint32_t sok = 0;
#pragma unroll
    for (int q = 0; q < kLPL; ++q) {
        const int s = lane + 32 * q;
        tail[q] = (s < G && nc[q] == uint32_t(C)) ? __ldcg(&rr[s].cand[C - 1]) : 0ull;
    }
#pragma unroll
    for (int t = 0; t < kSPL; ++t) {
        const int j = lane + 32 * t;
        sk[t] = 0u;
        if (j < ns) {
            const int s = j / h, i = j - s * h;
            const uint32_t n_s = __ldcg(&rr[s].nc);
            const unsigned long long w = __ldcg(&rr[s].cand[i]);
            if (uint32_t(i) < n_s) {
                sk[t] = cand_key(w);
                sok |= 1u << t;
            }
        }
    }
    bool overflow = false;
    unsigned long long tau_inc = 0ull;  // tokens missing from every list lie below it
#pragma unroll
    for (int q = 0; q < kLPL; ++q) {
        overflow |= nc[q] == kOverflow;
        tau_inc = tail[q] > tau_inc ? tail[q] : tau_inc;
    }
    if (__any_sync(0xffffffffu, overflow)) {
        fallback = true;
        return -1;
    }
    tau_inc = warp_max_u64(tau_inc);
    const int nvalid = __reduce_add_sync(0xffffffffu, __popc(sok));
    // every word whose value reaches the C-th sampled value: the row's top C and ties
    const uint32_t vt = nvalid >= C ? warp_kth_key<kSPL>(sk, sok, C) : 0u;
    const int n0 = gather_lists(rr, G, nc, vt, buf, 0);
    if (n0 > kBufCap || n0 == 0) {
        fallback = true;
        return -1;
    }
    sort_buf(buf, n0);
    const int lim = min(n0, kKeepCap);
    const int nk = small_k ? min(ri.k, n0) : lim;
    const int iA = lane, iB = lane + 32;
    const unsigned long long cA = iA < lim ? buf[iA] : 0ull;
    const unsigned long long cB = iB < lim ? buf[iB] : 0ull;
    const float xA = key2f(cand_key(cA)), xB = key2f(cand_key(cB));
    const int idxA = cand_idx(cA), idxB = cand_idx(cB);
    auto complete = [&](int i) { return i < 0 || buf[i] >= tau_inc; };
    int np = nk;
    if (ri.do_topp) {
        // prefix masses in fp32; redone in double when a prefix lies near the cut
        const float eA = iA < nk ? __expf((xA - m) * ri.invT) : 0.0f;
        const float eB = iB < nk ? __expf((xB - m) * ri.invT) : 0.0f;
        float sA = eA, sB = eB;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float oA = __shfl_up_sync(0xffffffffu, sA, off);
            const float oB = __shfl_up_sync(0xffffffffu, sB, off);
            if (lane >= off) {
                sA += oA;
                sB += oB;
            }
        }
        sB += __shfl_sync(0xffffffffu, sA, 31);
        float Z;
        if (small_k) {
            Z = __shfl_sync(0xffffffffu, sB, 31);
        } else {
            float z = 0.0f;
            for (int s = lane; s < G; s += 32) {
                const float mxs = __ldcg(&rr[s].mx);
                if (!(mxs > -INFINITY)) continue;
                const float zs = __ldcg(&rr[s].zs) - __ldcg(&rr[s].zc);
                z += zs * __expf((mxs - m) * ri.invT);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
            Z = z;
        }
        const float pz = ri.p * Z;
        const float exA = sA - eA, exB = sB - eB;
        const float tol = 1e-4f * Z;
        const bool nearcut = __any_sync(0xffffffffu, (iA < nk && fabsf(exA - pz) < tol) ||
                                                         (iB < nk && fabsf(exB - pz) < tol));
        if (!nearcut) {
            const bool kA = iA < nk && (exA < pz || iA == 0);
            const bool kB = iB < nk && (exB < pz);
            np = __popc(__ballot_sync(0xffffffffu, kA)) + __popc(__ballot_sync(0xffffffffu, kB));
        } else {
            // close to the cut: the same walk in double
            const double Te = double(ri.Te);
            const double y0 = double(m) / Te;
            const double dA = iA < nk ? exp(double(xA) / Te - y0) : 0.0;
            const double dB = iB < nk ? exp(double(xB) / Te - y0) : 0.0;
            double qA = dA, qB = dB;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double oA = __shfl_up_sync(0xffffffffu, qA, off);
                const double oB = __shfl_up_sync(0xffffffffu, qB, off);
                if (lane >= off) {
                    qA += oA;
                    qB += oB;
                }
            }
            qB += __shfl_sync(0xffffffffu, qA, 31);
            double ZD;
            if (small_k) {
                ZD = __shfl_sync(0xffffffffu, qB, 31);
            } else {
                double z = 0.0;
                for (int s = lane; s < G; s += 32) {
                    const float mxs = __ldcg(&rr[s].mx);
                    if (!(mxs > -INFINITY)) continue;
                    const double zs = double(__ldcg(&rr[s].zs)) - double(__ldcg(&rr[s].zc));
                    z += zs * exp((double(mxs) - double(m)) / Te);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
                ZD = z;
            }
            const double pzd = double(ri.p) * ZD;
            const bool kA = iA < nk && ((qA - dA) < pzd || iA == 0);
            const bool kB = iB < nk && ((qB - dB) < pzd);
            np = __popc(__ballot_sync(0xffffffffu, kA)) + __popc(__ballot_sync(0xffffffffu, kB));
        }
        if (!small_k && np >= lim) fallback = true;
    } else if (!small_k) {
        np = lim;
    }
    int nkept = np;
    if (ri.do_minp) {
        const double th = double(m) + double(ri.Te) * log(double(ri.minp));
        float xthr = float(th);
        if (double(xthr) < th) xthr = nextafterf(xthr, INFINITY);
        const bool mA = iA < np && xA >= xthr;
        const bool mB = iB < np && xB >= xthr;
        nkept = __popc(__ballot_sync(0xffffffffu, mA)) + __popc(__ballot_sync(0xffffffffu, mB));
        nkept = max(nkept, 1);
        if (!small_k && !ri.do_topp && nkept >= lim) fallback = true;
    } else if (!small_k && !ri.do_topp) {
        fallback = true;
    }
    if (!fallback) {
        // every kept token must be known exactly, and so must the first dropped
        // one when min-p or top-p (not top-k) closed the set
        if (!complete(nkept - 1)) fallback = true;
        if (small_k && !complete(nk - 1)) fallback = true;
        if (nkept < (small_k ? nk : lim) && !complete(nkept)) fallback = true;
    }
    if (!fallback) {
        GTop2 t;
        t.a = grec_empty();
        t.b = grec_empty();
        if (iA < nkept) top2_insert(t, cand_grec(ri, xA, idxA));
        if (iB < nkept) top2_insert(t, cand_grec(ri, xB, idxB));
        top2_warp_reduce(t);
        token = settle_fast(t, ri.T);
    }
    __syncwarp();
    return token;
}

// Finish row r from its records (one warp). Returns 1 when the row needs the
// CTA-wide exact path (m and amax are returned for it), 0 otherwise. Loads of
// the G <= kMaxUnits records are issued together (kLPL per lane).
__device__ __noinline__ int finish_row(const ColParams& P, unsigned long long* buf, const int r,
                                       const RowInfo ri, float* m_out, int* amax_out)
{
    const int lane = threadIdx.x & 31;
    const KernelParams& kp = P.k;
    const int G = P.gc;
    const ColRec* rr = P.rec + int64_t(r) * G;
    __threadfence();

    uint4 hd[kLPL];
    GTop2 t;
    t.a = grec_empty();
    t.b = grec_empty();
    const bool plain = ri.cls == kClsPlain;
#pragma unroll
    for (int q = 0; q < kLPL; ++q) {
        const int s = lane + 32 * q;
        hd[q] = s < G ? __ldcg(reinterpret_cast<const uint4*>(&rr[s]))  // mx, amax, flags, nc
                      : make_uint4(0xFF800000u, uint32_t(INT_MAX), 0u, 0u);
        if (plain && s < G) {
            const uint4 ua = __ldcg(reinterpret_cast<const uint4*>(&rr[s].g0));
            const uint4 ub = __ldcg(reinterpret_cast<const uint4*>(&rr[s].g1));
            top2_insert(t, GRec{__uint_as_float(ua.x), int(ua.y), __uint_as_float(ua.z), ua.w});
            top2_insert(t, GRec{__uint_as_float(ub.x), int(ub.y), __uint_as_float(ub.z), ub.w});
        }
    }
    float m = -INFINITY;
    int am = INT_MAX;
    uint32_t fl = 0;
    uint32_t nc[kLPL];
#pragma unroll
    for (int q = 0; q < kLPL; ++q) {
        fl |= hd[q].z;
        maxidx_merge(m, am, __uint_as_float(hd[q].x), int(hd[q].y));
        nc[q] = hd[q].w;
    }
    warp_maxidx(m, am);
    fl = __reduce_or_sync(0xffffffffu, fl);
    int status = ri.status;
    if (status == kRowOk) {
        if (fl & kFlagNonFinite) status = kRowNonFinite;
        else if (!(fl & kFlagAnyFinite)) status = kRowAllNegInf;
    }
    *m_out = m;
    *amax_out = am;
    int token = -1;
    bool fallback = false;
    if (status != kRowOk) {
        token = -1;
    } else if (ri.cls == kClsGreedy) {
        token = am;
    } else if (plain) {
        top2_warp_reduce(t);
        token = settle_fast(t, ri.T);
    } else {
        token = finish_cand(P, buf, ri, rr, nc, m, fallback);
    }
    if (lane == 0) {
        if (!fallback) {
            kp.out_tokens[r] = token;
            if (kp.out_status) kp.out_status[r] = status;
        }
        P.counters[r] = 0u;
    }
    return fallback ? 1 : 0;
}

// ---------------------------------------------------------------- one unit
template <typename InT>
__device__ __forceinline__ void unit_step(const ColParams& P, ColShared& sh, int uid, uint4* slot,
                                          unsigned long long* buf)
{
    const KernelParams& kp = P.k;
    const int lane = threadIdx.x & 31;
    Unit u;
    u.r = uid / P.gc;
    u.s = uid - u.r * P.gc;
    u.v0 = u.s * P.w;
    int lrow = u.r;
    if (kp.logit_row) lrow = kp.logit_row[u.r];
    const bool lrow_ok = lrow >= 0 && int64_t(lrow) < kp.n_logit_rows;
    u.n = lrow_ok ? max(0, min(P.w, int(kp.vocab) - u.v0)) : 0;
    stage_unit<InT>(kp, lrow_ok ? lrow : 0, u, slot);
    const RowInfo ri = load_row_info(P, u.r, lrow_ok ? lrow : -1);
    ColRec* rec = P.rec + int64_t(u.r) * P.gc + u.s;
    if (ri.cls == kClsGreedy) {
        unit_greedy<InT>(u, slot, rec);
    } else if (ri.cls == kClsPlain) {
        unit_plain<InT>(u, ri, slot, rec);
    } else if (ri.cls == kClsCand) {
        unit_cand<InT>(u, ri, slot, buf, rec);
    } else {
        cp_async_wait<0>();
        if (lane == 0) {
            rec->mx = -INFINITY;
            rec->amax = INT_MAX;
            rec->flags = kFlagAnyFinite;
            rec->nc = 0;
        }
    }
    // the record is complete once every lane has written its part; lane 0's
    // release publishes all of it
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atom_add_release_gpu(&P.counters[u.r], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == uint32_t(P.gc - 1)) {
        float mrow;
        int arow;
        const int fb = finish_row(P, buf, u.r, ri, &mrow, &arow);
        if (fb && lane == 0) {
            const int q = atomicAdd(&sh.n_fallback, 1);
            sh.fallback_rows[q] = u.r;
            sh.fb_m[q] = mrow;
            sh.fb_amax[q] = arow;
        }
    }
    __syncwarp();
}

template <typename InT>
__global__ void __launch_bounds__(kT, 1) colsplit_kernel(const ColParams P)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    ColShared& sh = *reinterpret_cast<ColShared*>(smem_raw);
    const int tid = threadIdx.x, wid = tid >> 5;
    unsigned char* wbase = smem_raw + kSharedHead + size_t(wid) * kWarpBytes;
    uint4* slot = reinterpret_cast<uint4*>(wbase);
    unsigned long long* buf = reinterpret_cast<unsigned long long*>(wbase + kSlotBytes);
    if (tid == 0) sh.n_fallback = 0;
    __syncthreads();
#pragma unroll 1
    for (int u = blockIdx.x + gridDim.x * wid; u < P.n_units; u += gridDim.x * kW)
        unit_step<InT>(P, sh, u, slot, buf);
    __syncthreads();

    // ---- rows the lists could not settle: exact path, whole CTA
    const int nf = sh.n_fallback;
    if (tid == 0 && nf > 0 && P.stats) atomicAdd(&P.stats[0], (unsigned long long)nf);
    for (int q = 0; q < nf; ++q) {
        const int r = sh.fallback_rows[q];
        int lrow = r;
        if (P.k.logit_row) lrow = P.k.logit_row[r];
        const RowInfo ri = load_row_info(P, r, lrow);
        cta_exact_row<InT>(sh, P, r, ri, sh.fb_m[q], sh.fb_amax[q]);
    }
}

}  // namespace col
}  // namespace dst
