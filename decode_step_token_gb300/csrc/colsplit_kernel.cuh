// colsplit_kernel.cuh -- body of the column-split kernel (design in colsplit.cuh).
//
// Per CTA: warps pull rows from a shared queue. Each warp keeps a ring of three
// staged rows in shared memory: while it works on one row, 16-byte asynchronous
// copies (cp.async) bring its slices of the next two rows and their parameters.
// For each row the warp writes the (row, slice) record from lane 0 and
// publishes it with a release atomic on the row's counter; the counter's old
// value is examined one row later, and the warp that completed the count
// finishes the row. Loops over a slice's vectors stay rolled, which keeps the
// hot code small.
#pragma once

#include <cuda_bf16.h>

#include "colsplit.cuh"

namespace dst {
namespace col {

__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t* p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gsrc)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------- staging a row
// Bring row r's parameters and this CTA's slice of its logits into a ring slot
// (all lanes of the warp). Tokens past the slice end are staged as -inf.
template <typename InT>
__device__ __forceinline__ void stage_row(const ColParams& P, int r, SlotHdr* hdr, uint4* vec, int v0, int n)
{
    constexpr int ES = int(sizeof(InT));
    constexpr int EPV = ElemTraits<InT>::kPerVec;
    const KernelParams& kp = P.k;
    const int lane = threadIdx.x & 31;
    int lrow = r;
    if (kp.logit_row) lrow = kp.logit_row[r];
    const bool lrow_ok = lrow >= 0 && int64_t(lrow) < kp.n_logit_rows;
    switch (lane) {
        case 0: cp_async4(&hdr->T, kp.temperature + r); break;
        case 1: if (kp.top_k) cp_async4(&hdr->k, kp.top_k + r); else hdr->k = -1; break;
        case 2: if (kp.top_p) cp_async4(&hdr->p, kp.top_p + r); else hdr->p = 1.0f; break;
        case 3: if (kp.min_p) cp_async4(&hdr->minp, kp.min_p + r); else hdr->minp = 0.0f; break;
        case 4: if (kp.stream_id) cp_async4(&hdr->stream_id, kp.stream_id + r); break;
        case 5: if (kp.seed) cp_async8(&hdr->seed_lo, kp.seed + r); break;
        case 6: hdr->lrow = lrow_ok ? lrow : -1; hdr->r = r; break;
        case 7: if (kp.presence) cp_async4(&hdr->pres, kp.presence + r); else hdr->pres = 0.0f; break;
        case 8: if (kp.frequency) cp_async4(&hdr->freq, kp.frequency + r); else hdr->freq = 0.0f; break;
        case 9: if (kp.repetition) cp_async4(&hdr->rep, kp.repetition + r); else hdr->rep = 1.0f; break;
        case 10:
            // cp.async moves 4 bytes at least: fetch the aligned word holding the byte
            if (kp.has_seed) {
                const uintptr_t a = reinterpret_cast<uintptr_t>(kp.has_seed + r);
                cp_async4(&hdr->has_seed, reinterpret_cast<const void*>(a & ~uintptr_t(3)));
                hdr->hs_shift = int(a & 3u) * 8;
            } else {
                hdr->has_seed = 0u;
                hdr->hs_shift = 0;
            }
            break;
        default: break;
    }
    if (!lrow_ok || n <= 0) return;
    const unsigned char* g = static_cast<const unsigned char*>(kp.logits) + (int64_t(lrow) * kp.row_stride + v0) * ES;
    const int nfull = n / EPV, nvec = (n + EPV - 1) / EPV;
    const bool aligned = (reinterpret_cast<uintptr_t>(g) & 15u) == 0;
    if (aligned)
        for (int j = lane; j < nfull; j += 32) cp_async16(vec + j, g + 16 * size_t(j));
    // vectors not copied whole: built from plain loads, padded with -inf
    for (int j = (aligned ? nfull : 0) + lane; j < nvec; j += 32) {
        InT e[EPV];
#pragma unroll
        for (int q = 0; q < EPV; ++q) {
            const int i = j * EPV + q;
            if (sizeof(InT) == 2) {
                uint16_t b = 0xFF80u;  // bf16 -inf
                if (i < n) b = reinterpret_cast<const uint16_t*>(g)[i];
                reinterpret_cast<uint16_t*>(e)[q] = b;
            } else {
                float f = -INFINITY;
                if (i < n) f = reinterpret_cast<const float*>(g)[i];
                reinterpret_cast<float*>(e)[q] = f;
            }
        }
        vec[j] = *reinterpret_cast<const uint4*>(e);
    }
}

// Validate and classify a staged row.
__device__ __forceinline__ RowInfo finalize_row(const ColParams& P, const SlotHdr& h, int r)
{
    const KernelParams& kp = P.k;
    const int64_t V = kp.vocab;
    RowInfo ri;
    ri.T = h.T;
    ri.k = h.k;
    ri.p = h.p;
    ri.minp = h.minp;
    const bool seeded = ((h.has_seed >> h.hs_shift) & 0xFFu) != 0u;
    const uint64_t key = seeded ? ((uint64_t(h.seed_hi) << 32) | h.seed_lo) : kp.global_seed;
    const uint32_t sid = kp.stream_id ? h.stream_id : (seeded ? 0u : uint32_t(r));
    ri.stream = (sid & 0x7FFFFFFFu) | (seeded ? 0x80000000u : 0u);
    ri.key_lo = uint32_t(key);
    ri.key_hi = uint32_t(key >> 32);
    ri.lrow = h.lrow < 0 ? 0 : h.lrow;
    bool bad = h.lrow < 0;
    if (!(ri.T >= 0.0f) || isinf(ri.T)) bad = true;
    if (!(ri.k == -1 || ri.k >= 1)) bad = true;
    if (!(ri.p > 0.0f && ri.p <= 1.0f)) bad = true;
    if (!(ri.minp >= 0.0f && ri.minp <= 1.0f)) bad = true;
    if (!isfinite(h.pres) || !isfinite(h.freq)) bad = true;
    if (!(h.rep > 0.0f) || isinf(h.rep)) bad = true;
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

// The same, straight from global memory (the exact path, rare).
__device__ __noinline__ RowInfo global_row_info(const ColParams& P, int r)
{
    const KernelParams& kp = P.k;
    SlotHdr h;
    int lrow = kp.logit_row ? kp.logit_row[r] : r;
    h.lrow = (lrow >= 0 && int64_t(lrow) < kp.n_logit_rows) ? lrow : -1;
    h.T = kp.temperature[r];
    h.k = kp.top_k ? kp.top_k[r] : -1;
    h.p = kp.top_p ? kp.top_p[r] : 1.0f;
    h.minp = kp.min_p ? kp.min_p[r] : 0.0f;
    h.stream_id = kp.stream_id ? kp.stream_id[r] : 0u;
    const uint64_t sd = kp.seed ? kp.seed[r] : 0ull;
    h.seed_lo = uint32_t(sd);
    h.seed_hi = uint32_t(sd >> 32);
    h.has_seed = kp.has_seed ? uint32_t(kp.has_seed[r]) : 0u;
    h.hs_shift = 0;
    h.pres = kp.presence ? kp.presence[r] : 0.0f;
    h.freq = kp.frequency ? kp.frequency[r] : 0.0f;
    h.rep = kp.repetition ? kp.repetition[r] : 1.0f;
    return finalize_row(P, h, r);
}

// ln E for E = -ln(u), 1 - u = w, from lg2(w); |error| < 2e-5, enough to rank
// candidates (the final comparison is redone in double).
__device__ __forceinline__ float fast_ln_exp1(float w, float lg2w, uint32_t word)
{
    // small w: -ln(1 - w) = w (1 + w/2 + w^2/3 + ...), so ln E = ln w + w/2 + 5w^2/24 + w^3/8
    const float series = fmaf(lg2w, 0.69314718055994531f, w * fmaf(w, fmaf(w, 0.125f, 0.20833333f), 0.5f));
    const float direct = __logf(-__logf(noise_u(word)));
    return w < 0.03125f ? series : direct;
}

// ---------------------------------------------------------------- per-class slice summaries
// Vector helpers: the 8 (bf16) or 4 (fp32) logits of a 16-byte vector.
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
        const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
        // NaN propagates through additions (an inf - inf NaN implies a +inf, itself an error)
        const __nv_bfloat162 sm = __hadd2(__hadd2(a, b), __hadd2(c, d));
        const float s0 = __low2float(sm), s1 = __high2float(sm);
        nan = (s0 != s0) || (s1 != s1);
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
        const float sm = (a + b) + (c + d);
        nan = sm != sm;
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

struct MaxAcc {
    float mx;
    int am;
    bool nan;
};

// Lane max / argmax (lowest index on ties) over the staged slice: one comparison
// chain step per vector.
template <typename InT>
__device__ __forceinline__ MaxAcc lane_max(const uint4* vec, int v0, int nvec)
{
    constexpr int EPV = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    MaxAcc a{-INFINITY, INT_MAX, false};
#pragma unroll 2
    for (int j = lane; j < nvec; j += 32) {
        const uint4 raw = vec[j];
        bool nan;
        const float m = Vec<InT>::vmax(raw, nan);
        a.nan |= nan;
        if (m > a.mx) {
            a.mx = m;
            a.am = v0 + j * EPV + vec_find<InT>(raw, m);
        }
    }
    return a;
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

template <typename InT>
__device__ __noinline__ void summarize_plain(const RowInfo ri, const uint4* vec, int v0, int n, ColRec* rec)
{
    constexpr int EPV = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const int nvec = (n + EPV - 1) / EPV;
    const float invT = ri.invT;
    const float a2 = invT * 1.4426950408889634f;
    const PhiloxKey key{ri.key_lo, ri.key_hi};
    const uint32_t stream = ri.stream, olo = ri.off_lo, ohi = ri.off_hi;
    // seed the entry bar with the lane's largest logit: the winner is rarely far below it
    const MaxAcc mx = lane_max<InT>(vec, v0, nvec);
    PlainAcc a;
    a.best = grec_empty();
    a.c2 = INFINITY;
    if (mx.mx > -INFINITY && mx.mx <= 3.402823466e38f) {
        const uint4 blk = philox4x32_10(make_uint4(uint32_t(mx.am) >> 2, stream, olo, ohi), key);
        plain_take(a, invT, mx.am, mx.mx, lane_of(blk, uint32_t(mx.am) & 3u));
    }
#pragma unroll 1
    for (int j = lane; j < nvec; j += 32) {
        const int vb = v0 + j * EPV;  // a multiple of 4
        const uint4 raw = vec[j];
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
        for (int e = 0; e < EPV; ++e) {
            xs[e] = Vec<InT>::get(raw, e);
            // the score is at most x/T - ln(1 - u): only tokens that may beat the bar
            const float lg2w = __log2f(noise_one_minus_u(ws[e]));
            mask |= (fmaf(xs[e], a2, a.c2) > lg2w) ? (1u << e) : 0u;
        }
        while (mask) {
            const int e = __ffs(mask) - 1;
            mask &= mask - 1;
            const int v = vb + e;
            if (v != a.best.idx) plain_take(a, invT, v, pickf<EPV>(xs, e), picku<EPV>(ws, e));
        }
    }
    GTop2 t;
    t.a = a.best;
    t.b = grec_empty();
    top2_warp_reduce(t);
    const bool bad = __any_sync(0xffffffffu, mx.nan || mx.mx > 3.402823466e38f);
    const bool fin = t.a.idx != INT_MAX;
    if (lane == 0) {
        rec->mx = 0.0f;
        rec->amax = 0;
        rec->flags = (bad ? kFlagNonFinite : 0u) | (fin ? kFlagAnyFinite : 0u);
        rec->nc = 0;
        rec->g0 = t.a;
        rec->g1 = t.b;
    }
}

template <typename InT>
__device__ __noinline__ void summarize_max(const RowInfo ri, const uint4* vec, int v0, int n, ColRec* rec,
                                           unsigned long long* buf, bool candidates)
{
    constexpr int EPV = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const int nvec = (n + EPV - 1) / EPV;
    const MaxAcc a = lane_max<InT>(vec, v0, nvec);
    const float lane_mx = a.mx;
    float mx = a.mx;
    int am = a.am;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, off);
        const int oi = __shfl_xor_sync(0xffffffffu, am, off);
        maxidx_merge(mx, am, om, oi);
    }
    const bool bad = __any_sync(0xffffffffu, a.nan) || mx > 3.402823466e38f;
    const bool fin = mx > -INFINITY && !(mx > 3.402823466e38f);
    uint32_t nc = 0;
    unsigned long long my_cand = 0ull;  // lane l < 8 holds candidate l
    float zs = 0.0f, zc = 0.0f;
    if (candidates) {
        // tau = the 8th largest lane maximum: at least 8 tokens of the slice reach it
        int rk = 0;
        for (int l = 0; l < 32; ++l) {
            const float o = __shfl_sync(0xffffffffu, lane_mx, l);
            rk += (o > lane_mx) || (o == lane_mx && l < lane);
        }
        const unsigned bal = __ballot_sync(0xffffffffu, rk == kSliceCand - 1);
        const float tau = __shfl_sync(0xffffffffu, lane_mx, bal ? __ffs(bal) - 1 : 0);
        int cnt = 0;
#pragma unroll 1
        for (int j0 = 0; j0 < nvec; j0 += 32) {
            const int j = j0 + lane;
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (j < nvec) raw = vec[j];
            const int vb = v0 + j * EPV;
            uint32_t mask = 0;
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const float x = Vec<InT>::get(raw, e);
                mask |= (j < nvec && vb + e < v0 + n && x >= tau) ? (1u << e) : 0u;
                if (ri.need_z && j < nvec && x > -INFINITY) {
                    const float y = __expf((x - mx) * ri.invT) - zc;
                    const float s2 = zs + y;
                    zc = (s2 - zs) - y;
                    zs = s2;
                }
            }
            if (__any_sync(0xffffffffu, mask != 0)) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    const bool take = (mask >> e) & 1u;
                    const unsigned bt = __ballot_sync(0xffffffffu, take);
                    if (take) {
                        const int pos = cnt + __popc(bt & ((1u << lane) - 1u));
                        if (pos < 64) buf[pos] = comp_of(Vec<InT>::get(raw, e), vb + e);
                    }
                    cnt += __popc(bt);
                }
            }
        }
        __syncwarp();
        if (cnt > 64) {
            nc = kOverflow;
        } else {
            unsigned long long ca = lane < cnt ? buf[lane] : 0ull;
            unsigned long long cb = lane + 32 < cnt ? buf[lane + 32] : 0ull;
            warp_sort64_desc(ca, cb);
            nc = uint32_t(min(cnt, kSliceCand));
            my_cand = lane < int(nc) ? ca : 0ull;
        }
        if (ri.need_z) {
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
        __syncwarp();
    }
    // lane 0 writes the whole record, so its release atomic publishes all of it
    unsigned long long c[kSliceCand];
#pragma unroll
    for (int l = 0; l < kSliceCand; ++l) c[l] = __shfl_sync(0xffffffffu, my_cand, l);
    if (lane == 0) {
        rec->mx = mx;
        rec->amax = am;
        rec->flags = (bad ? kFlagNonFinite : 0u) | (fin ? kFlagAnyFinite : 0u);
        rec->nc = nc;
        if (candidates) {
#pragma unroll
            for (int l = 0; l < kSliceCand; ++l) rec->cand[l] = c[l];
            rec->zs = zs;
            rec->zc = zc;
        }
    }
}

// ---------------------------------------------------------------- finishing a row
// Pick between the two best fp32 Gumbel candidates; double precision only when
// they are within fp32 reach of each other.
__device__ __forceinline__ int settle_fast(const GTop2& t, float T)
{
    if (t.a.idx == INT_MAX) return -1;
    if (t.b.idx == INT_MAX) return t.a.idx;
    const float tol = 1e-4f + 1e-5f * fmaxf(fabsf(t.a.s), fabsf(t.b.s));
    if (t.a.s - t.b.s > tol) return t.a.idx;
    return settle_top2(t, T);
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

// Finish row r from its records (one warp). Returns 1 when the row needs the
// CTA-wide exact path (m and amax are returned for it), 0 otherwise.
__device__ __noinline__ int finish_row(const ColParams& P, unsigned long long* scratch, const int r,
                                       const RowInfo ri, float* m_out, int* amax_out)
{
    const int lane = threadIdx.x & 31;
    const KernelParams& kp = P.k;
    const int G = P.gc;
    const ColRec* rr = P.rec + int64_t(r) * G;
    __threadfence();

    float m = -INFINITY;
    int am = INT_MAX;
    uint32_t fl = 0;
    for (int s = lane; s < G; s += 32) {
        const uint4 h = __ldcg(reinterpret_cast<const uint4*>(&rr[s]));  // mx, amax, flags, nc
        fl |= h.z;
        maxidx_merge(m, am, __uint_as_float(h.x), int(h.y));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, off);
        const int oi = __shfl_xor_sync(0xffffffffu, am, off);
        maxidx_merge(m, am, om, oi);
        fl |= __shfl_xor_sync(0xffffffffu, fl, off);
    }
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
    } else if (ri.cls == kClsPlain) {
        GTop2 t;
        t.a = grec_empty();
        t.b = grec_empty();
        for (int s = lane; s < G; s += 32) {
            const uint4 ua = __ldcg(reinterpret_cast<const uint4*>(&rr[s].g0));
            const uint4 ub = __ldcg(reinterpret_cast<const uint4*>(&rr[s].g1));
            const GRec a{__uint_as_float(ua.x), int(ua.y), __uint_as_float(ua.z), ua.w};
            const GRec b{__uint_as_float(ub.x), int(ub.y), __uint_as_float(ub.z), ub.w};
            top2_insert(t, a);
            top2_insert(t, b);
        }
        top2_warp_reduce(t);
        token = settle_fast(t, ri.T);
    } else {
        // ---- truncated row: merge the slices' candidates
        const bool small_k = ri.small_k;
        if (ri.do_topk && !small_k) fallback = true;
        unsigned long long tau_inc = 0ull;  // below this the merged list may miss tokens
        bool overflow = false;
        uint32_t hk[kMaxGcPerLane];
#pragma unroll
        for (int t = 0; t < kMaxGcPerLane; ++t) {
            const int s = lane + 32 * t;
            hk[t] = 0u;
            if (s < G) {
                const uint32_t nc = __ldcg(&rr[s].nc);
                if (nc == kOverflow) {
                    overflow = true;
                } else {
                    if (nc >= 1u) hk[t] = cand_key(__ldcg(&rr[s].cand[0]));
                    if (nc == uint32_t(kSliceCand)) {
                        const unsigned long long c7 = __ldcg(&rr[s].cand[kSliceCand - 1]);
                        tau_inc = c7 > tau_inc ? c7 : tau_inc;
                    }
                }
            }
        }
        overflow = __any_sync(0xffffffffu, overflow);
        tau_inc = warp_max_u64(tau_inc);
        fallback = fallback || overflow;
        unsigned long long* buf = scratch;
        int n0 = 0;
        if (!fallback) {
            // K0: the largest key with at least L slice heads at or above it
            const int L = small_k ? ri.k : kKeepCap;
            uint32_t K0 = 0;
            if (G >= L) {
                uint32_t lo = 0, hi = 0xFFFFFFFFu;  // invariant: count(key >= lo) >= L
                while (lo < hi) {
                    const uint32_t mid = lo + (hi - lo) / 2 + 1;
                    int c = 0;
#pragma unroll
                    for (int t = 0; t < kMaxGcPerLane; ++t) c += hk[t] >= mid ? 1 : 0;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
                    if (c >= L) lo = mid;
                    else hi = mid - 1;
                }
                K0 = lo;
            }
            // gather every submitted candidate with key >= K0
            for (int s0 = 0; s0 < G; s0 += 32) {
                const int s = s0 + lane;
                const uint32_t nc = s < G ? __ldcg(&rr[s].nc) : 0u;
                for (int c = 0; c < kSliceCand; ++c) {
                    unsigned long long w = 0ull;
                    if (c < int(nc)) w = __ldcg(&rr[s].cand[c]);
                    const bool take = c < int(nc) && cand_key(w) >= K0;
                    const unsigned bt = __ballot_sync(0xffffffffu, take);
                    if (take) {
                        const int pos = n0 + __popc(bt & ((1u << lane) - 1u));
                        if (pos < kListCap) buf[pos] = w;
                    }
                    n0 += __popc(bt);
                }
            }
            if (n0 > kListCap || n0 == 0) fallback = true;
        }
        if (!fallback) {
            warp_sort_smem_desc(buf, n0);
            const int lim = min(n0, kKeepCap);
            const int nk = small_k ? min(ri.k, n0) : lim;
            const int iA = lane, iB = lane + 32;
            const unsigned long long cA = iA < lim ? buf[iA] : 0ull;
            const unsigned long long cB = iB < lim ? buf[iB] : 0ull;
            const float xA = key2f(cand_key(cA)), xB = key2f(cand_key(cB));
            const int idxA = cand_idx(cA), idxB = cand_idx(cB);
            auto complete = [&](int i) { return i < 0 || buf[i] > tau_inc; };
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
        }
        __syncwarp();
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

template <typename InT>
__device__ __forceinline__ void summarize(const RowInfo& ri, const uint4* vec, int v0, int n, ColRec* rec,
                                          unsigned long long* buf)
{
    if (ri.cls == kClsPlain) {
        summarize_plain<InT>(ri, vec, v0, n, rec);
    } else if (ri.cls == kClsErr) {
        if ((threadIdx.x & 31) == 0) {
            rec->mx = -INFINITY;
            rec->amax = INT_MAX;
            rec->flags = kFlagAnyFinite;
            rec->nc = 0;
        }
    } else {
        summarize_max<InT>(ri, vec, v0, n, rec, buf, ri.cls == kClsCand);
    }
}

template <typename InT, int NV>
__global__ void __launch_bounds__(kT, 1) colsplit_kernel(const ColParams P)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    ColShared& sh = *reinterpret_cast<ColShared*>(smem_raw);
    constexpr int EPV = ElemTraits<InT>::kPerVec;
    constexpr int kVecBytes = NV * 32 * 16 > kListCap * 8 ? NV * 32 * 16 : kListCap * 8;
    constexpr int kSlotBytes = int(sizeof(SlotHdr)) + kVecBytes;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int s = blockIdx.x;
    const int N = P.n_rows;
    const int V = int(P.k.vocab);
    const int v0 = s * P.w;
    const int n = max(0, min(V - v0, P.w));
    unsigned char* ring = smem_raw + ((sizeof(ColShared) + 127) & ~size_t(127)) +
                          size_t(wid) * kSlots * kSlotBytes;
    auto hdr_of = [&](int slot) { return reinterpret_cast<SlotHdr*>(ring + slot * kSlotBytes); };
    auto vec_of = [&](int slot) { return reinterpret_cast<uint4*>(ring + slot * kSlotBytes + sizeof(SlotHdr)); };
    if (tid == 0) {
        sh.next_row = 0;
        sh.n_fallback = 0;
        sh.offset = P.k.philox_offset_dev ? *P.k.philox_offset_dev : P.k.philox_offset;
    }
    __syncthreads();
    const uint32_t off_lo = uint32_t(sh.offset), off_hi = uint32_t(sh.offset >> 32);

    auto pop = [&]() {
        int r = 0;
        if (lane == 0) r = atomicAdd(&sh.next_row, 1);
        return __shfl_sync(0xffffffffu, r, 0);
    };

    int r0 = pop();
    if (r0 < N) stage_row<InT>(P, r0, hdr_of(0), vec_of(0), v0, n);
    cp_async_commit();
    int r1 = pop();
    if (r1 < N) stage_row<InT>(P, r1, hdr_of(1), vec_of(1), v0, n);
    cp_async_commit();
    int cur = 0;
    int pend_r = -1;
    RowInfo pend_ri;
    uint32_t pend_old = 0;
    auto finish_pending = [&](unsigned long long* scratch) {
        const uint32_t old = __shfl_sync(0xffffffffu, pend_old, 0);
        if (old != uint32_t(P.gc - 1)) return;
        float mrow;
        int arow;
        const int fb = finish_row(P, scratch, pend_r, pend_ri, &mrow, &arow);
        if (fb && lane == 0) {
            const int q = atomicAdd(&sh.n_fallback, 1);
            sh.fallback_rows[q] = pend_r;
            sh.fb_m[q] = mrow;
            sh.fb_amax[q] = arow;
        }
        __syncwarp();
    };
    while (true) {
        const int r2 = pop();
        const int slot2 = cur == 0 ? 2 : cur - 1;
        if (r2 < N) stage_row<InT>(P, r2, hdr_of(slot2), vec_of(slot2), v0, n);
        cp_async_commit();
        cp_async_wait<2>();
        __syncwarp();
        if (r0 >= N) break;
        RowInfo ri = finalize_row(P, *hdr_of(cur), r0);
        ri.off_lo = off_lo;
        ri.off_hi = off_hi;
        ColRec* rec = P.rec + int64_t(r0) * P.gc + s;
        unsigned long long* scratch = reinterpret_cast<unsigned long long*>(vec_of(cur));
        summarize<InT>(ri, vec_of(cur), v0, ri.status == kRowOk ? n : 0, rec, scratch);
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = atom_add_release_gpu(&P.counters[r0], 1u);
        if (pend_r >= 0) finish_pending(scratch);
        pend_r = r0;
        pend_ri = ri;
        pend_old = old;
        r0 = r1;
        r1 = r2;
        cur = cur == 2 ? 0 : cur + 1;
    }
    cp_async_wait<0>();
    __syncwarp();
    if (pend_r >= 0) finish_pending(reinterpret_cast<unsigned long long*>(vec_of(cur)));
    __syncthreads();

    // ---- rows the candidates could not settle: exact path, whole CTA
    const int nf = sh.n_fallback;
    if (tid == 0 && nf > 0 && P.stats) atomicAdd(&P.stats[0], (unsigned long long)nf);
    for (int q = 0; q < nf; ++q) {
        RowInfo ri = global_row_info(P, sh.fallback_rows[q]);
        ri.off_lo = off_lo;
        ri.off_hi = off_hi;
        cta_exact_row<InT>(sh, P, sh.fallback_rows[q], ri, sh.fb_m[q], sh.fb_amax[q]);
    }
    (void)EPV;
}

}  // namespace col
}  // namespace dst
