// colsplit_kernel.cuh -- body of the unit-split kernel (design in colsplit.cuh).
//
// Per warp and unit: the unit's logits go to the warp's shared-memory slot by
// 16-byte cp.async copies in kStages commit groups, the row's parameters are
// read while they fly, and the class pass (greedy / plain / truncated) starts on
// the first group as soon as it has landed. Loops stay rolled and every pass is
// out-of-line: code that a warp runs once per launch is fetched cold, so it is
// kept short.
#pragma once

#include <cuda_bf16.h>

#include "colsplit.cuh"

namespace dst {
namespace col {

static_assert(kStages == 4, "wait_stage below spells out four stages");

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
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

// Hardware log2 of a positive normal fp32 value (flush-to-zero form: the inputs
// here are draws >= 2^-24 and their logs, never denormal).
__device__ __forceinline__ float lg2_ftz(float x)
{
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// log2 of E = -ln(u) for the draw of word `word`, branch-free: for 1 - u < 1/32 the
// series of fast_ln_exp1 (in log2 units), else log2(-log2 u) + log2(ln 2).
__device__ __forceinline__ float log2_exp1(uint32_t word)
{
    const float w = noise_one_minus_u(word);
    const float lw = lg2_ftz(w);
    const float series = w * fmaf(w, fmaf(w, 0.125f, 0.20833333f), 0.5f) * 1.4426950408889634f + lw;
    const float direct = lg2_ftz(-lg2_ftz(noise_u(word))) - 0.52876637294489771f;
    return w < 0.03125f ? series : direct;
}

template <typename InT>
__device__ __forceinline__ uint4 neg_inf_vec()
{
    const uint32_t w = sizeof(InT) == 2 ? 0xFF80FF80u : 0xFF800000u;
    return make_uint4(w, w, w, w);
}

// Gumbel-max over the unit, scores x/T - ln E in log2 units. A bound with one log2
// per token filters against the warp's best; vectors with a surviving token are
// scored exactly by the whole warp at once (a per-lane slow path would diverge).
// The Philox blocks of a vector come from the row-folded generator.
template <typename InT>
__device__ __noinline__ void unit_plain(const Unit u, const RowInfo ri, const uint4* slot, ColRec* rec)
{
    constexpr int EPV = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const float invT = ri.invT;
    const float a2 = invT * 1.4426950408889634f;
    const RowPhilox ph = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, ri.off_lo, ri.off_hi);
    float c2 = INFINITY;  // minus the bar, log2 units: +inf until the warp has a best
    float best2 = -INFINITY, bx = 0.0f;
    int bi = INT_MAX;
    uint32_t bw = 0;
    float lm = -INFINITY;
    bool nan = false;
#pragma unroll 1
    for (int st = 0; st < kStages; ++st) {
        wait_stage(st);
        const int e = min((st + 1) * u.q, u.nvec);
        // a token can beat the warp's best only if x/T - ln(1 - u) clears it (E >= 1 - u):
        // one log2 per token decides; a vector where any lane has such a token is
        // scored exactly by the whole warp (a uniform branch), which also lifts the bar
        // the loop is warp-uniform (every lane runs every step; lanes past the end see
        // -inf) because the step holds warp-wide votes and shuffles
#pragma unroll 1
        for (int j0 = st * u.q; j0 < e; j0 += 32) {
            const int j = j0 + lane;
            const uint4 raw = j < e ? slot[j] : neg_inf_vec<InT>();
            const int vb = u.v0 + j * EPV;  // a multiple of 4: the vector's blocks start at vb / 4
            bool vn;
            lm = fmaxf(lm, Vec<InT>::vmax(raw, vn));
            nan |= vn;
            uint32_t ws[EPV];
#pragma unroll
            for (int b = 0; b < EPV / 4; ++b) {
                const uint4 blk = philox_block(ph, uint32_t(vb >> 2) + uint32_t(b));
                ws[4 * b + 0] = blk.x;
                ws[4 * b + 1] = blk.y;
                ws[4 * b + 2] = blk.z;
                ws[4 * b + 3] = blk.w;
            }
            bool pass = false;
#pragma unroll
            for (int q = 0; q < EPV; ++q)
                pass |= fmaf(Vec<InT>::get(raw, q), a2, c2) > lg2_ftz(noise_one_minus_u(ws[q]));
            if (__any_sync(0xffffffffu, pass)) {
#pragma unroll
                for (int q = 0; q < EPV; ++q) {
                    const float s2 = fmaf(Vec<InT>::get(raw, q), a2, -log2_exp1(ws[q]));
                    if (s2 > best2) {  // tokens come in increasing order: ties keep the first
                        best2 = s2;
                        bi = vb + q;
                    }
                }
                float wb = best2;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) wb = fmaxf(wb, __shfl_xor_sync(0xffffffffu, wb, off));
                // bar: the warp's best less the margin of the final comparison (log2 units)
                if (wb > -INFINITY) c2 = -(wb - (1e-4f + 1e-6f * fabsf(wb * 0.69314718055994531f)) * 1.4426950408889634f);
            }
        }
    }
    // the lane's winner: its logit and Philox word once more
    if (bi != INT_MAX) {
        const int jb = (bi - u.v0) / EPV, qb = (bi - u.v0) % EPV;
        const uint4 rb = slot[jb];
        bx = Vec<InT>::get(rb, qb);
        bw = lane_of(philox_block(ph, uint32_t(bi) >> 2), uint32_t(bi) & 3u);
    }
    const uint32_t flags = unit_flags(lm, nan);
    GTop2 t;
    t.a = bi != INT_MAX ? GRec{best2 * 0.69314718055994531f, bi, bx, bw} : grec_empty();
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

// ---------------------------------------------------------------- truncated units
// The unit's top-C list (C = k for k <= 64, else 64), sorted by (value desc,
// index asc): each lane deals its vectors to GPL groups in turn (GPL = 1, 2 or 4
// as C needs), tau = the C-th largest of the 32 GPL group maxima -- found by a
// bitwise search counted with warp ballots -- is reached by at least C of the
// unit's tokens, so the unit's top C are among the tokens >= tau, which are
// gathered and sorted.
template <int GPL>
__device__ __forceinline__ uint32_t kth_group_max(const float (&g)[GPL], int C)
{
    // the largest key K with at least C group maxima >= K, one bit at a time from
    // the top: each step counts the qualifying maxima of the warp with ballots
    uint32_t key[GPL];
#pragma unroll
    for (int a = 0; a < GPL; ++a) key[a] = f2key(g[a]);
    uint32_t K = 0;
#pragma unroll 1
    for (int b = 31; b >= 0; --b) {
        const uint32_t cand = K | (1u << b);
        int n = 0;
#pragma unroll
        for (int a = 0; a < GPL; ++a) n += __popc(__ballot_sync(0xffffffffu, key[a] >= cand));
        if (n >= C) K = cand;
    }
    return K;
}

template <typename InT, int GPL>
__device__ __forceinline__ void unit_cand_impl(const Unit u, const RowInfo ri, const uint4* slot,
                                               unsigned long long* buf, ColRec* rec)
{
    constexpr int EPV = Vec<InT>::E;
    const int lane = threadIdx.x & 31;
    const int C = ri.small_k ? ri.k : kCandCap;
    float mx = -INFINITY;
    float g[GPL];
#pragma unroll
    for (int a = 0; a < GPL; ++a) g[a] = -INFINITY;
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
            // this vector joins group 0, then the groups rotate
            const float gn = fmaxf(g[0], m);
#pragma unroll
            for (int a = 0; a + 1 < GPL; ++a) g[a] = g[a + 1];
            g[GPL - 1] = gn;
        }
    }
    const uint32_t flags = unit_flags(mx, nan);
    warp_maxidx(mx, am);
    const uint32_t tauk = kth_group_max<GPL>(g, C);
    const float tau = key2f(tauk);
    // tokens >= tau (finite), each lane into its own kSeg words of buf (word i of
    // lane l at buf[32 i + l]); and, for top-p without top-k, the unit's mass
    int my = 0;
    float zs = 0.0f, zc = 0.0f;
    const bool need_z = ri.need_z;
    const float invT = ri.invT;
#pragma unroll 1
    for (int j = lane; j < u.nvec; j += 32) {
        const uint4 raw = slot[j];
        const int vb = u.v0 + j * EPV;
        if (need_z) {
#pragma unroll
            for (int q = 0; q < EPV; ++q) {
                const float x = Vec<InT>::get(raw, q);
                if (x > -INFINITY) {
                    const float y = __expf((x - mx) * invT) - zc;
                    const float s2 = zs + y;
                    zc = (s2 - zs) - y;
                    zs = s2;
                }
            }
        } else {
            bool vn;
            if (!(Vec<InT>::vmax(raw, vn) >= tau)) continue;  // no token of the vector qualifies
        }
        uint32_t mask = 0;
#pragma unroll
        for (int q = 0; q < EPV; ++q) {
            const float x = Vec<InT>::get(raw, q);
            mask |= (x >= tau && x > -INFINITY) ? (1u << q) : 0u;
        }
        while (mask) {
            const int q = __ffs(mask) - 1;
            mask &= mask - 1;
            if (my < kSeg) buf[32 * my + lane] = comp_of(Vec<InT>::get(raw, q), vb + q);
            ++my;
        }
    }
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
    int pre = my;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, pre, off);
        if (lane >= off) pre += o;
    }
    const int cnt = __shfl_sync(0xffffffffu, pre, 31);
    pre -= my;
    uint32_t nc;
    if (__any_sync(0xffffffffu, my > kSeg) || cnt > kUnitCands) {
        nc = kOverflow;  // the row takes the exact path
    } else {
        // the unit's logits are no longer needed: pack the words into the slot, sort
        unsigned long long* dst = reinterpret_cast<unsigned long long*>(const_cast<uint4*>(slot));
        __syncwarp();
        for (int i = 0; i < my; ++i) dst[pre + i] = buf[32 * i + lane];
        __syncwarp();
        warp_sort_smem_desc(dst, cnt);
        nc = uint32_t(min(cnt, C));
        for (int i = lane; i < int(nc); i += 32) rec->cand[i] = dst[i];
    }
    if (lane == 0) {
        rec->mx = mx;
        rec->amax = am;
        rec->flags = flags;
        rec->nc = nc;
        rec->zs = zs;
        rec->zc = zc;
        rec->tau = tauk;
    }
    __syncwarp();
}

template <typename InT>
__device__ __noinline__ void unit_cand(const Unit u, const RowInfo ri, const uint4* slot,
                                       unsigned long long* buf, ColRec* rec)
{
    const int C = ri.small_k ? ri.k : kCandCap;
    if (C <= 16) unit_cand_impl<InT, 1>(u, ri, slot, buf, rec);
    else if (C <= 32) unit_cand_impl<InT, 2>(u, ri, slot, buf, rec);
    else unit_cand_impl<InT, 4>(u, ri, slot, buf, rec);
}

// ---------------------------------------------------------------- one unit (phase 1)
template <typename InT>
__device__ __forceinline__ void unit_step(const ColParams& P, int uid, uint4* slot, unsigned long long* buf)
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
    // the record is complete: count the unit in (release after the warp's writes)
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        atomicAdd(&P.sync->done[u.r], 1u);
    }
}

// ---------------------------------------------------------------- row readiness
constexpr uint32_t kBarPolls = 1u << 24;  // about a second of polling

// The whole CTA waits until all G units of row r have written their records; the
// records are then visible to every thread of the CTA. Returns false if the wait
// gave up (the state is then marked broken for later launches).
__device__ __noinline__ bool wait_row(ColShared& sh, RowSync* sync, int r, int G)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        if (ld_acquire_gpu(&sync->poison) != 0u) {
            ok = 0;
        } else {
            uint32_t polls = 0;
            while (ld_acquire_gpu(&sync->done[r]) < uint32_t(G)) {
                if (++polls > kBarPolls) {
                    ok = 0;
                    atomicExch(&sync->poison, 1u);
                    break;
                }
                if (polls > 64) __nanosleep(32);
            }
        }
        sh.bar_ok = ok;
    }
    __syncthreads();
    return sh.bar_ok != 0;
}

// ---------------------------------------------------------------- phase 2
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

// Finish a greedy, plain or rejected row r from its records (one warp). Loads
// of the G <= kMaxUnits records are issued together (kLPL per lane).
__device__ __noinline__ void finish_row(const ColParams& P, const int r, const RowInfo ri)
{
    const int lane = threadIdx.x & 31;
    const KernelParams& kp = P.k;
    const int G = P.gc;
    const ColRec* rr = P.rec + int64_t(r) * G;
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
#pragma unroll
    for (int q = 0; q < kLPL; ++q) {
        fl |= hd[q].z;
        maxidx_merge(m, am, __uint_as_float(hd[q].x), int(hd[q].y));
    }
    warp_maxidx(m, am);
    fl = __reduce_or_sync(0xffffffffu, fl);
    int status = ri.status;
    if (status == kRowOk) {
        if (fl & kFlagNonFinite) status = kRowNonFinite;
        else if (!(fl & kFlagAnyFinite)) status = kRowAllNegInf;
    }
    int token = -1;
    if (status != kRowOk) {
        token = -1;
    } else if (ri.cls == kClsGreedy) {
        token = am;
    } else {
        top2_warp_reduce(t);
        token = settle_fast(t, ri.T);
    }
    if (lane == 0) {
        kp.out_tokens[r] = token;
        if (kp.out_status) kp.out_status[r] = status;
    }
}

// Number of the first nk sorted tokens (x, two per lane: index lane and
// lane + 32) kept by top-p, walked in double: for cuts that fp32 cannot call.
__device__ __noinline__ int topp_keep_f64(const RowInfo ri, float xA, float xB, int nk, float m, bool small_k,
                                          const float* hmx, const float* hzs, const float* hzc, int G)
{
    const int lane = threadIdx.x & 31;
    const int iA = lane, iB = lane + 32;
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
            if (!(hmx[s] > -INFINITY)) continue;
            z += (double(hzs[s]) - double(hzc[s])) * exp((double(hmx[s]) - double(m)) / Te);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        ZD = z;
    }
    const double pzd = double(ri.p) * ZD;
    const bool kA = iA < nk && ((qA - dA) < pzd || iA == 0);
    const bool kB = iB < nk && ((qB - dB) < pzd);
    return __popc(__ballot_sync(0xffffffffu, kA)) + __popc(__ballot_sync(0xffffffffu, kB));
}

// Smallest fp32 x with x >= m + T ln(min_p) in exact arithmetic.
__device__ __noinline__ float minp_threshold(float m, float Te, float minp)
{
    const double th = double(m) + double(Te) * log(double(minp));
    float xthr = float(th);
    if (double(xthr) < th) xthr = nextafterf(xthr, INFINITY);
    return xthr;
}

// The kept set of a truncated row from L[0, n): the largest tokens of the
// units' lists by (value desc, index asc), sorted; every token missing from the
// lists lies below tau_inc, so L[i] is the row's i-th token when L[i] >= tau_inc.
// Warp 0 only. Returns the token, or sets `fallback` when the list cannot
// settle it.
__device__ __forceinline__ int cut_and_pick(const RowInfo ri, const unsigned long long* L, int n,
                                         unsigned long long tau_inc, float m, const float* hmx,
                                         const float* hzs, const float* hzc, int G, bool& fallback)
{
    const int lane = threadIdx.x & 31;
    const bool small_k = ri.small_k;
    const int lim = min(n, kKeepCap);
    const int nk = small_k ? min(ri.k, n) : lim;
    const int iA = lane, iB = lane + 32;
    const unsigned long long cA = iA < lim ? L[iA] : 0ull;
    const unsigned long long cB = iB < lim ? L[iB] : 0ull;
    const float xA = key2f(cand_key(cA)), xB = key2f(cand_key(cB));
    const int idxA = cand_idx(cA), idxB = cand_idx(cB);
    auto complete = [&](int i) { return i < 0 || L[i] >= tau_inc; };
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
            for (int s = lane; s < G; s += 32)
                if (hmx[s] > -INFINITY) z += (hzs[s] - hzc[s]) * __expf((hmx[s] - m) * ri.invT);
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
            np = topp_keep_f64(ri, xA, xB, nk, m, small_k, hmx, hzs, hzc, G);
        }
        if (!small_k && np >= lim) fallback = true;  // the set may run past the list
    } else if (!small_k) {
        np = lim;
    }
    int nkept = np;
    if (ri.do_minp) {
        const float xthr = minp_threshold(m, ri.Te, ri.minp);
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
    int token = -1;
    if (!fallback) {
        // exact fp32 scores (log2 units) of the lane's two candidates, their Philox
        // blocks taken together from the row-folded generator
        const RowPhilox ph = row_philox(PhiloxKey{ri.key_lo, ri.key_hi}, ri.stream, ri.off_lo, ri.off_hi);
        const uint4 bA = philox_block(ph, uint32_t(idxA) >> 2);
        const uint4 bB = philox_block(ph, uint32_t(idxB) >> 2);
        const uint32_t wA = lane_of(bA, uint32_t(idxA) & 3u), wB = lane_of(bB, uint32_t(idxB) & 3u);
        const float a2 = ri.invT * 1.4426950408889634f;
        const float sA = iA < nkept ? fmaf(xA, a2, -log2_exp1(wA)) : -INFINITY;
        const float sB = iB < nkept ? fmaf(xB, a2, -log2_exp1(wB)) : -INFINITY;
        const int jA = iA < nkept ? idxA : INT_MAX, jB = iB < nkept ? idxB : INT_MAX;
        // the warp's best two (score desc, token asc): a warp maximum, then another
        // without the winner
        const bool aFirst = sA > sB || (sA == sB && jA < jB);
        float s1 = aFirst ? sA : sB, s2 = aFirst ? sB : sA;
        int i1 = aFirst ? jA : jB, i2 = aFirst ? jB : jA;
        float bs = s1;
        int bi = i1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, bs, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (os > bs || (os == bs && oi < bi)) {
                bs = os;
                bi = oi;
            }
        }
        float cs = i1 == bi ? s2 : s1;  // this lane's best apart from the winner
        int ci = i1 == bi ? i2 : i1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, cs, off);
            const int oi = __shfl_xor_sync(0xffffffffu, ci, off);
            if (os > cs || (os == cs && oi < ci)) {
                cs = os;
                ci = oi;
            }
        }
        token = bi == INT_MAX ? -1 : bi;
        const float n1 = bs * 0.69314718055994531f, n2 = cs * 0.69314718055994531f;
        const float tol = 1e-4f + 1e-5f * fmaxf(fabsf(n1), fabsf(n2));
        if (bi != INT_MAX && ci != INT_MAX && !(n1 - n2 > tol)) {
            // within fp32 reach: settle the pair in double from their logits and words
            GTop2 t;
            t.a = grec_empty();
            t.b = grec_empty();
            const unsigned ha = __ballot_sync(0xffffffffu, jA == bi || jB == bi);
            const unsigned hb = __ballot_sync(0xffffffffu, jA == ci || jB == ci);
            const int la = __ffs(ha) - 1, lb = __ffs(hb) - 1;
            const float xa = __shfl_sync(0xffffffffu, jA == bi ? xA : xB, la);
            const uint32_t wa = __shfl_sync(0xffffffffu, jA == bi ? wA : wB, la);
            const float xb = __shfl_sync(0xffffffffu, jA == ci ? xA : xB, lb);
            const uint32_t wb = __shfl_sync(0xffffffffu, jA == ci ? wA : wB, lb);
            t.a = GRec{n1, bi, xa, wa};
            t.b = GRec{n2, ci, xb, wb};
            token = settle_fast(t, ri.T);
        }
    }
    return token;
}

// Finish truncated row r with the whole CTA. One round of copies brings every
// unit's sorted top list and header into shared memory. t1 = the C-th largest of
// the lists' first h words (G h >= C) bounds the row's top C from below, so the
// listed words >= t1 hold them; those are gathered, ranked, and warp 0 cuts and
// picks. `dyn` is the CTA's free dynamic shared memory.
__device__ __noinline__ void cta_cand_row(ColShared& sh, const ColParams& P, int r, const RowInfo ri,
                                          unsigned char* dyn)
{
    const KernelParams& kp = P.k;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int G = P.gc;
    const int C = ri.small_k ? ri.k : kCandCap;
    unsigned long long* Lst = reinterpret_cast<unsigned long long*>(dyn);  // [G][kCandCap]
    unsigned long long* S = Lst + size_t(kMaxUnits) * kCandCap;            // gathered
    unsigned long long* Out = S + kSelCap;                                  // ranked
    uint32_t* rank = reinterpret_cast<uint32_t*>(Out + kSelCap);
    float* hmx = reinterpret_cast<float*>(rank + kSelCap);
    float* hzs = hmx + kMaxUnits;
    float* hzc = hzs + kMaxUnits;
    uint32_t* hnc = reinterpret_cast<uint32_t*>(hzc + kMaxUnits);
    int32_t* ham = reinterpret_cast<int32_t*>(hnc + kMaxUnits);
    uint32_t* hfl = reinterpret_cast<uint32_t*>(ham + kMaxUnits);
    const ColRec* rr = P.rec + int64_t(r) * G;
    const int pieces = (C + 1) / 2;  // 16-byte pieces of a list
    for (int c = tid; c < G * pieces; c += kT) {
        const int s = c / pieces, h = c - s * pieces;
        cp_async16(Lst + s * kCandCap + 2 * h, &rr[s].cand[2 * h]);
    }
    cp_async_commit();
    if (tid < G) {
        const uint4 hd = __ldcg(reinterpret_cast<const uint4*>(&rr[tid]));  // mx, amax, flags, nc
        hmx[tid] = __uint_as_float(hd.x);
        ham[tid] = int(hd.y);
        hfl[tid] = hd.z;
        hnc[tid] = hd.w;
        const uint4 hz = __ldcg(reinterpret_cast<const uint4*>(&rr[tid].zs));  // zs, zc, tau, pad
        hzs[tid] = __uint_as_float(hz.x);
        hzc[tid] = __uint_as_float(hz.y);
    }
    if (tid == 0) sh.n_sel = 0;
    cp_async_wait<0>();
    __syncthreads();
    if (wid == 0) {
        float m = -INFINITY;
        int am = INT_MAX;
        uint32_t fl = 0, over = 0;
        unsigned long long ti = 0ull;  // tokens missing from every list lie below it
        for (int s = lane; s < G; s += 32) {
            maxidx_merge(m, am, hmx[s], ham[s]);
            fl |= hfl[s];
            over |= hnc[s] == kOverflow ? 1u : 0u;
            if (hnc[s] == uint32_t(C)) ti = max(ti, Lst[s * kCandCap + C - 1]);
        }
        warp_maxidx(m, am);
        fl = __reduce_or_sync(0xffffffffu, fl);
        over = __reduce_or_sync(0xffffffffu, over);
        ti = warp_max_u64(ti);
        if (lane == 0) {
            sh.fin_m = m;
            sh.fin_amax = am;
            sh.fin_flags = fl;
            sh.fin_over = over;
            sh.fin_tinc = ti;
        }
    }
    __syncthreads();
    const float m = sh.fin_m;
    const int am = sh.fin_amax;
    int status = ri.status;
    if (status == kRowOk) {
        if (sh.fin_flags & kFlagNonFinite) status = kRowNonFinite;
        else if (!(sh.fin_flags & kFlagAnyFinite)) status = kRowAllNegInf;
    }
    bool fallback = status == kRowOk && (sh.fin_over != 0 || (ri.do_topk && !ri.small_k));
    int n = 0;
    if (status == kRowOk && !fallback) {
        // samples: the first h words of every list
        const int h = min(C, (C + G - 1) / G);
        for (int e = tid; e < G * h; e += kT) {
            const int s = e / h, i = e - s * h;
            if (uint32_t(i) < hnc[s]) S[atomicAdd(&sh.n_sel, 1)] = Lst[s * kCandCap + i];
        }
        __syncthreads();
        const int ns = sh.n_sel;  // <= G h < G + C <= kSelCap
        unsigned long long t1 = 0ull;
        if (ns >= C) {
            cta_rank_sort_desc(S, ns, rank, Out);
            t1 = Out[C - 1];
        }
        __syncthreads();
        if (tid == 0) sh.n_sel = 0;
        __syncthreads();
        for (int e = tid; e < G * kCandCap; e += kT) {
            const int s = e / kCandCap, i = e - s * kCandCap;
            if (uint32_t(i) < hnc[s] && Lst[e] >= t1) {
                const int pos = atomicAdd(&sh.n_sel, 1);
                if (pos < kSelCap) S[pos] = Lst[e];
            }
        }
        __syncthreads();
        n = sh.n_sel;
        if (n > kSelCap || n == 0) fallback = true;
        else cta_rank_sort_desc(S, n, rank, Out);
    }
    if (wid == 0) {
        int token = -1;
        if (status == kRowOk && !fallback)
            token = cut_and_pick(ri, Out, n, sh.fin_tinc, m, hmx, hzs, hzc, G, fallback);
        if (lane == 0) {
            if (fallback) {
                const int q = atomicAdd(&sh.n_fallback, 1);
                sh.fallback_rows[q] = r;
                sh.fb_m[q] = m;
                sh.fb_amax[q] = am;
            } else {
                kp.out_tokens[r] = token;
                if (kp.out_status) kp.out_status[r] = status;
            }
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- the kernel
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

    // ---- phase 1: units, dealt so that consecutive CTAs take consecutive units
#pragma unroll 1
    for (int u = blockIdx.x + gridDim.x * wid; u < P.n_units; u += gridDim.x * kW)
        unit_step<InT>(P, u, slot, buf);

    // ---- phase 2: rows, dealt round-robin to the CTAs; each waits for its own units
    const KernelParams& kp = P.k;
#pragma unroll 1
    for (int r = blockIdx.x; r < P.n_rows; r += gridDim.x) {
        const bool ok = wait_row(sh, P.sync, r, P.gc);
        int lrow = r;
        if (kp.logit_row) lrow = kp.logit_row[r];
        const bool lrow_ok = lrow >= 0 && int64_t(lrow) < kp.n_logit_rows;
        const RowInfo ri = load_row_info(P, r, lrow_ok ? lrow : -1);
        if (!ok) {
            if (tid == 0) {
                kp.out_tokens[r] = -1;
                if (kp.out_status) kp.out_status[r] = kRowTimeout;
            }
        } else if (ri.cls == kClsCand) {
            cta_cand_row(sh, P, r, ri, smem_raw + kSharedHead);
        } else if (wid == 0) {
            finish_row(P, r, ri);
        }
        // the row's records are read: zero its counter for the next launch
        __syncthreads();
        if (tid == 0 && ok) P.sync->done[r] = 0u;
    }
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
