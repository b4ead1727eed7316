// group_sampler_kernel.cuh -- the kernel body (see group_sampler.cuh for the design).
#pragma once

#include "group_sampler.cuh"

namespace dst {
namespace grp {

__device__ __forceinline__ float nan_f() { return __int_as_float(0x7fc00000); }

// Fork classes decided from the parameters alone (every CTA decides alike).
__device__ __forceinline__ bool fork_truncates(const RowParams& rp)
{
    return rp.do_topk || rp.do_topp || rp.do_minp;
}

// The fork needs the softmax mass of the whole row at its temperature: top-p whose
// domain the thread maxima cannot bound by top-k, or outputs over every token.
__device__ __forceinline__ bool fork_needs_z(const RowParams& rp, int n_tmax)
{
    if (rp.status != kRowOk) return false;
    if (rp.do_topp && !(rp.do_topk && rp.k <= n_tmax)) return true;
    return rp.want_out && !fork_truncates(rp);
}

// Add one token to digit d of the exact path's histograms. Lanes of a warp that
// hit the same digit are combined first (one atomic per digit and warp): the
// leading digits of nearby values coincide, and same-address atomics serialise.
__device__ __forceinline__ void hist_add(GShared& sh, uint32_t d, unsigned long long w, bool mass_mode)
{
    const unsigned active = __activemask();
    const unsigned peers = __match_any_sync(active, d);
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(peers) - 1;
    if (mass_mode) {
        unsigned long long sum = 0;
        unsigned rest = peers;
        while (rest) {
            const int j = __ffs(rest) - 1;
            rest &= rest - 1;
            sum += __shfl_sync(peers, w, j);
        }
        if (lane == leader) atomicAdd(&sh.hmass[d], sum);
    }
    if (lane == leader) atomicAdd(&sh.hcnt[d], uint32_t(__popc(peers)));
}

// Cluster-wide selection of the kept prefix in (value desc, index asc) order over
// the staged row: the first token whose inclusive weight (1 per token, or the
// fixed-point softmax mass) reaches the target closes the prefix. Tokens outside
// the domain prefix (dkey, didx) weigh nothing. Every CTA of the cluster calls it.
template <typename InT>
__device__ void exact_select(GShared& sh, const Part& pt, const RowParams& rp, uint32_t rank, uint32_t C,
                             bool mass_mode, bool dom, uint32_t dkey, int didx, float m,
                             unsigned long long count_target, uint32_t& out_key, int& out_idx)
{
    const int tid = threadIdx.x;
    if (tid == 0) {
        sh.sel.prefix = 0;
        sh.sel.pbits = 0;
        sh.sel.w_above = 0;
        sh.sel.target = count_target;
        sh.sel.tie_cta = -1;
        sh.sel.tie_j = 0;
        sh.sel.bidx = 0;
    }
    __syncthreads();
    for (int level = 0; level < 4; ++level) {
        for (int i = tid; i < 256; i += kT) {
            sh.hcnt[i] = 0;
            sh.hmass[i] = 0;
        }
        __syncthreads();
        const uint32_t prefix = sh.sel.prefix, pbits = sh.sel.pbits;
        const int shift = 24 - 8 * level;
        part_for_each<InT>(pt, rp, [&](int v, float x) {
            const uint32_t key = f2key(x);
            if (dom && !in_prefix(key, v, dkey, didx)) return;
            if (pbits && (key >> (32 - pbits)) != prefix) return;
            const uint32_t d = (key >> shift) & 255u;
            hist_add(sh, d, mass_mode ? mass_q(x, m, rp.invT) : 0ull, mass_mode);
        });
        __syncthreads();
        cluster_sync();
        if (rank == 0) {
            const int d = tid;  // one thread per digit (kT == 256)
            unsigned long long tc = 0, tm = 0;
            for (uint32_t c = 0; c < C; ++c) {
                tc += dsmem_ld_u32(dsmem_map(smem_addr(&sh.hcnt[d]), c));
                if (mass_mode) tm += dsmem_ld_u64(dsmem_map(smem_addr(&sh.hmass[d]), c));
            }
            const unsigned long long wgt = mass_mode ? tm : tc;
            // inclusive suffix sum over digits (this digit and all larger ones)
            const int lane = tid & 31, wid = tid >> 5;
            unsigned long long s = wgt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned long long o = __shfl_down_sync(0xffffffffu, s, off);
                if (lane + off < 32) s += o;
            }
            if (lane == 0) sh.red_q[wid] = s;
            __syncthreads();
            unsigned long long later = 0, total = 0;
            for (int w = 0; w < kW; ++w) {
                if (w > wid) later += sh.red_q[w];
                total += sh.red_q[w];
            }
            const unsigned long long incl = s + later;
            unsigned long long target = sh.sel.target;
            if (mass_mode && level == 0) {
                target = (unsigned long long)ceil(double(rp.p) * double(total));
                if (target < 1) target = 1;
            }
            const unsigned long long above = incl - wgt;
            const unsigned long long wa = sh.sel.w_above;
            __syncthreads();
            if (tid == 0) sh.sel.target = target;
            if (wa + incl >= target && wa + above < target) {
                const uint32_t np = (prefix << 8) | uint32_t(d);
                const unsigned long long nwa = wa + above;
                sh.sel.prefix = np;
                sh.sel.pbits = pbits + 8;
                sh.sel.w_above = nwa;
                if (level == 3) {
                    const unsigned long long wt = mass_mode ? mass_q(key2f(np), m, rp.invT) : 1ull;
                    const unsigned long long J = (target - nwa + wt - 1) / wt;
                    unsigned long long before = 0;
                    int cstar = int(C) - 1;
                    unsigned long long jloc = 0;
                    for (uint32_t c = 0; c < C; ++c) {
                        const unsigned long long cc = dsmem_ld_u32(dsmem_map(smem_addr(&sh.hcnt[d]), c));
                        if (J > before && J <= before + cc) {
                            cstar = int(c);
                            jloc = J - before;
                            break;
                        }
                        before += cc;
                    }
                    sh.sel.tie_cta = cstar;
                    sh.sel.tie_j = int(jloc);
                }
            }
            __syncthreads();
            if (tid < int(C)) dsmem_write(sh.sel, sh.sel, uint32_t(tid));
        }
        cluster_sync();
    }

    // the tie_j-th token (index order) carrying the boundary key
    const uint32_t K = sh.sel.prefix;
    if (int(rank) == sh.sel.tie_cta) {
        const int need = sh.sel.tie_j;
        int base = 0;
        for (int i0 = 0; i0 < pt.n; i0 += kT) {
            const int i = i0 + tid;
            int c = 0;
            if (i < pt.n) {
                const float x = part_x<InT>(pt, rp, i);
                const uint32_t key = f2key(x);
                c = (key == K && (!dom || in_prefix(key, pt.v0 + i, dkey, didx))) ? 1 : 0;
            }
            // exclusive scan of c over the block
            const int lane = tid & 31, wid = tid >> 5;
            int s = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += o;
            }
            __syncthreads();
            if (lane == 31) sh.red_i[wid] = s;
            __syncthreads();
            int before = 0, tot = 0;
            for (int w = 0; w < kW; ++w) {
                if (w < wid) before += sh.red_i[w];
                tot += sh.red_i[w];
            }
            const int excl = before + s - c;
            if (c && base + excl + 1 == need) {
                for (uint32_t cc = 0; cc < C; ++cc)
                    dsmem_st_u32(dsmem_map(smem_addr(&sh.sel.bidx), cc), uint32_t(pt.v0 + i));
            }
            base += tot;
            if (base >= need) break;
        }
    }
    cluster_sync();
    out_key = K;
    out_idx = sh.sel.bidx;
    __syncthreads();
}

}  // namespace grp
}  // namespace dst

namespace dst {
namespace grp {

__device__ __forceinline__ int block_min_i32(int v, GShared& sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
    __syncthreads();
    if (lane == 0) sh.red_i[wid] = v;
    __syncthreads();
    int t = INT_MAX;
#pragma unroll
    for (int w = 0; w < kW; ++w) t = min(t, sh.red_i[w]);
    return t;
}

// Bitonic sort of n words in shared memory, descending (n a power of two). Each
// warp owns n / 8 consecutive words: stages whose pairs stay inside one warp's
// words wait on that warp only; the others on the whole block.
template <typename T>
__device__ __noinline__ void block_sort_desc(T* a, int n)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int chunk = n / kW;
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const bool local = chunk >= 2 && stride < chunk;
            const int t0 = local ? wid * (chunk >> 1) + lane : threadIdx.x;
            const int t1 = local ? (wid + 1) * (chunk >> 1) : (n >> 1);
            const int step = local ? 32 : kT;
            for (int t = t0; t < t1; t += step) {
                const int lo = ((t & ~(stride - 1)) << 1) | (t & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const T x = a[lo], y = a[hi];
                if ((x < y) == desc) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            // the next stage may pair words across warps: wait for the block then
            const int nstride = stride > 1 ? stride >> 1 : size;
            const bool last = stride == 1 && size == n;
            const bool next_local = chunk >= 2 && nstride < chunk && !last;
            if (local && next_local) __syncwarp();
            else __syncthreads();
        }
    }
    __syncthreads();
}

// Inclusive prefix sum (thread order) of one 64-bit word per thread over the block.
__device__ __forceinline__ unsigned long long block_incl_scan_u64(unsigned long long v, GShared& sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long s = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += o;
    }
    __syncthreads();
    if (lane == 31) sh.red_q[wid] = s;
    __syncthreads();
    unsigned long long before = 0;
    for (int w = 0; w < wid; ++w) before += sh.red_q[w];
    return before + s;
}

// Leader CTA: the smallest thread maximum t such that the thread maxima >= t reach
// `target` -- a count, or their mass in units of 2^-20 of exp((x - m) / Te), each
// term rounded down -- or NaN when all of them fall short. Two rounds of 256 bins:
// on a log scale of the distance to m, then evenly inside the bin where the target
// is met. Bins only order the values (larger bin, smaller value).
// `bins` is 4 x 256 words of shared memory. The thread's maxima come by value
// (their first C entries): an array whose address reached this out-of-line
// function would live in local memory.
struct TmaxVals {
    float x[kMaxParts];
};
__device__ __noinline__ float tmax_select(GShared& sh, uint32_t* bins, const TmaxVals v, int C, float m, float tmin,
                                          bool mass, float invT, unsigned long long target)
{
    const int tid = threadIdx.x;
    uint32_t* bcnt = bins;
    uint32_t* bmin = bins + 256;
    uint32_t* bmax = bins + 512;
    uint32_t* bms = bins + 768;
    float lo = tmin, hi = m;
    unsigned long long pre = 0;
    // level-0 bin = 16 log2(1 + 64 (m - x) / (m - min maximum)): about 97 bins in all
    const float invT_bins = (m > tmin && m - tmin < INFINITY) ? 64.0f / (m - tmin) : 1.0f;
    for (int level = 0; level < 2; ++level) {
        bcnt[tid] = 0;
        bmin[tid] = 0xFFFFFFFFu;
        bmax[tid] = 0;
        bms[tid] = 0;
        __syncthreads();
        // level 0: bins on a log scale of the distance to m (heavy tails and narrow
        // rows alike spread over them); level 1: even bins inside the chosen bin
        const float inv = hi > lo ? 256.0f / (hi - lo) : 0.0f;
#pragma unroll
        for (int c = 0; c < kMaxParts; ++c) {
            const float x = v.x[c];
            if (c >= C || !(x > -INFINITY && x >= lo && x <= hi)) continue;
            const int bin = level == 0 ? min(255, int(__log2f(1.0f + (m - x) * invT_bins) * 16.0f))
                                       : min(255, max(0, int((hi - x) * inv)));
            const uint32_t key = f2key(x);
            atomicAdd(&bcnt[bin], 1u);
            atomicMin(&bmin[bin], key);
            atomicMax(&bmax[bin], key);
            if (mass) atomicAdd(&bms[bin], uint32_t(expf((x - m) * invT) * 1048576.0f));
        }
        __syncthreads();
        const unsigned long long w = mass ? (unsigned long long)bms[tid] : (unsigned long long)bcnt[tid];
        const unsigned long long cum = pre + block_incl_scan_u64(w, sh);
        const int first = block_min_i32(cum >= target ? tid : INT_MAX, sh);
        if (first == INT_MAX) return NAN;
        if (level == 1) {
            const uint32_t k = bmin[tid];
            const int kk = block_min_i32(tid <= first ? int(k ^ 0x80000000u) : INT_MAX, sh);
            return key2f(uint32_t(kk) ^ 0x80000000u);
        }
        // refine inside the first bin that meets the target
        if (tid == first) sh.red_q[0] = cum - w;
        __syncthreads();
        pre = sh.red_q[0];
        lo = key2f(bmin[first]);
        hi = key2f(bmax[first]);
        __syncthreads();
    }
    return NAN;
}

// Leader CTA: per truncating fork, a lower bound of its kept set from the thread
// maxima of the whole row (each is a token value of the row):
//   top-k: the smallest thread maximum that k or more thread maxima reach;
//   top-p: the smallest thread maximum t such that the thread maxima >= t alone,
//          less a rounding margin, carry p of the row's mass.
// `tk`/`tp` receive NaN where no bound exists.
__device__ __noinline__ void tmax_bounds(GShared& sh, uint32_t C, int g, float m, uint32_t* bins, float* tk,
                                         float* tp)
{
    const int tid = threadIdx.x;
    const int n = int(C) * kT;
    TmaxVals v;
    uint32_t kv[kMaxParts];
#pragma unroll
    for (int c = 0; c < kMaxParts; ++c)
        if (c < int(C)) kv[c] = dsmem_ld_u32(dsmem_map(smem_addr(&sh.tmax[tid]), uint32_t(c)));
    float lo = INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxParts; ++c) {
        v.x[c] = c < int(C) ? key2f(kv[c]) : -INFINITY;
        if (v.x[c] > -INFINITY) lo = fminf(lo, v.x[c]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    __syncthreads();
    if ((tid & 31) == 0) sh.red_f[tid >> 5] = lo;
    __syncthreads();
    float tmin = INFINITY;
    for (int w = 0; w < kW; ++w) tmin = fminf(tmin, sh.red_f[w]);
    for (int f = 0; f < g; ++f) {
        const RowParams& rp = sh.rp[f];
        const bool listed = sh.bc.f[f].kind == kKindList;
        const bool want_k = listed && rp.do_topk && rp.k <= n;
        const bool want_p = listed && rp.do_topp && !want_k;
        int twin_k = -1, twin_p = -1;
        for (int e = 0; e < f; ++e) {
            const RowParams& re = sh.rp[e];
            if (sh.bc.f[e].kind != kKindList) continue;
            if (want_k && re.do_topk && re.k == rp.k) twin_k = e;
            if (want_p && re.do_topp && !(re.do_topk && re.k <= n) && re.p == rp.p && re.invT == rp.invT &&
                sh.zrow[e] == sh.zrow[f])
                twin_p = e;
        }
        float rk = NAN, rpv = NAN;
        if (want_k) rk = twin_k >= 0 ? tk[twin_k] : tmax_select(sh, bins, v, int(C), m, tmin, false, 0.0f, (unsigned long long)rp.k);
        if (want_p) {
            if (twin_p >= 0) {
                rpv = tp[twin_p];
            } else {
                // fixed-point target, with a 1e-3 margin for the rounded fp32 terms
                const double t = double(rp.p) * sh.zrow[f] * 1048576.0 * 1.001;
                rpv = tmax_select(sh, bins, v, int(C), m, tmin, true, rp.invT, (unsigned long long)ceil(t));
            }
        }
        __syncthreads();
        if (tid == 0) {
            tk[f] = rk;
            tp[f] = rpv;
        }
        __syncthreads();
    }
}

// Sum over the staged part of exp((x - mc) / Te), compensated, as double.
template <typename InT>
__device__ __forceinline__ double part_mass(const Part& pt, const RowParams& rp, float mc, GShared& sh)
{
    // (x - mc) first: exact near the maximum, so tiny temperatures keep the top term at 1
    const float a2 = rp.invT * 1.4426950408889634f;
    float s = 0.0f, comp = 0.0f;
    part_for_each<InT>(pt, rp, [&](int, float x) {
        if (!(x > -INFINITY)) return;
        const float e = exp2f((x - mc) * a2);
        const float y = e - comp;
        const float t = s + y;
        comp = (t - s) - y;
        s = t;
    });
    return block_sum_f64(double(s) - double(comp), sh);
}

// The better of the two best fp32 Gumbel records: the fp32 order stands when the
// scores are further apart than fp32 rounding can reach; closer pairs are settled
// in double precision (slow on this GPU, so only then).
__device__ __forceinline__ int settle_pair(const GTop2& t, float T)
{
    if (t.a.idx == INT_MAX) return -1;
    if (t.b.idx == INT_MAX) return t.a.idx;
    const float tol = 1e-4f + 1e-5f * fmaxf(fabsf(t.a.s), fabsf(t.b.s));
    if (t.a.s - t.b.s > tol) return t.a.idx;
    return settle_top2(t, T);
}

// Copy the leader's group results into every CTA of the cluster, one word per thread.
__device__ __forceinline__ void bcast_cluster(GBcast& bc, uint32_t C)
{
    constexpr int kWords = int(sizeof(GBcast) / 4);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&bc);
    const uint32_t base = smem_addr(&bc);
    for (int w = threadIdx.x; w < kWords * int(C); w += kT) {
        const int c = w / kWords, i = w - c * kWords;
        if (c == 0) continue;  // the leader's own copy is the source
        dsmem_st_u32(dsmem_map(base + 4u * uint32_t(i), uint32_t(c)), src[i]);
    }
}

// Block-wide best two of one GTop2 per thread; the result is valid in thread 0.
__device__ __forceinline__ GTop2 block_top2(GTop2 t, GShared& sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    top2_warp_reduce(t);
    __syncthreads();
    if (lane == 0) sh.red_g[wid] = t;
    __syncthreads();
    GTop2 r;
    r.a = grec_empty();
    r.b = grec_empty();
    if (threadIdx.x == 0)
        for (int w = 0; w < kW; ++w) {
            top2_insert(r, sh.red_g[w].a);
            top2_insert(r, sh.red_g[w].b);
        }
    return r;
}

// Leader CTA: fork f's cut from the sorted candidate list, which holds every token
// of the row at or above the fork's bound tau: top-k, then top-p over the top-k
// domain, then min-p. Sets the last kept token as the fork's bound and kind Pick,
// or kind Exact when the list cannot settle the cut.
__device__ __noinline__ void resolve_cut(GShared& sh, const unsigned long long* list, int total, int f)
{
    const int tid = threadIdx.x;
    const RowParams& rp = sh.rp[f];
    ForkOut& fo = sh.bc.f[f];
    const float m = sh.bc.m;
    const uint32_t tkey = f2key(fo.tau);
    int c = 0;
    for (int i = tid; i < total; i += kT) c += cand_key(list[i]) >= tkey ? 1 : 0;
    const int nf = block_sum_i32(c, sh);

    const bool dom_complete = rp.do_topk && nf >= rp.k;
    const int dn = rp.do_topk ? min(rp.k, nf) : nf;
    bool unresolved = dn < 1;
    int np = dn;
    if (rp.do_topp && !unresolved) {
        // prefix masses in (value desc, index asc) order: fp32 terms, compensated
        // per thread over a run of consecutive entries, double across threads
        const int per = (dn + kT - 1) / kT;
        const int i0 = min(dn, tid * per), i1 = min(dn, i0 + per);
        float ls = 0.0f, lc = 0.0f;
        for (int i = i0; i < i1; ++i) {
            const float e = expf((key2f(cand_key(list[i])) - m) * rp.invT);
            const float y = e - lc;
            const float t = ls + y;
            lc = (t - ls) - y;
            ls = t;
        }
        const double loc = double(ls) - double(lc);
        double tot = 0.0;
        const double incl = block_incl_scan_f64(loc, sh, tot);
        double zdom = sh.zrow[f];
        if (rp.do_topk) {
            if (!dom_complete) unresolved = true;
            zdom = tot;
        }
        const double pz = double(rp.p) * zdom;
        int first = INT_MAX;
        double s = incl - loc;
        for (int i = i0; i < i1; ++i) {
            if (i > 0 && s >= pz) {
                first = i;
                break;
            }
            s += double(expf((key2f(cand_key(list[i])) - m) * rp.invT));
        }
        first = block_min_i32(first, sh);
        // the list holds every token >= tau; when tau is the min-p threshold, min-p
        // keeps at most the listed tokens, wherever the top-p cut falls beyond them
        const bool minp_caps = rp.do_minp && fo.tau <= fo.xthr;
        if (first != INT_MAX) np = first;
        else if (!dom_complete && tot < pz && !minp_caps) unresolved = true;
    } else if (rp.do_topk && !dom_complete && !(rp.do_minp && fo.tau <= fo.xthr)) {
        unresolved = true;
    }
    if (unresolved) {
        __syncthreads();
        if (tid == 0) fo.kind = kKindExact;
        __syncthreads();
        return;
    }
    int nk = np;
    if (rp.do_minp) {
        int b = INT_MAX;
        for (int i = tid; i < np; i += kT)
            if (key2f(cand_key(list[i])) < fo.xthr) b = min(b, i);
        b = block_min_i32(b, sh);
        nk = b == INT_MAX ? np : max(b, 1);
    }
    if (tid == 0) {
        const unsigned long long last = list[nk - 1];
        fo.bkey = cand_key(last);
        fo.bidx = cand_idx(last);
        fo.has_bound = 1;
        fo.kind = kKindPick;
        fo.listed = 1;
    }
    __syncthreads();
}

// Warp 0 of the leader: sort n <= 256 list words descending in registers and
// shuffles (word q * 32 + lane in v[q]; no block-wide waits), written back in place.
template <int PER>
__device__ __forceinline__ void warp_sort_words(unsigned long long* list, int n)
{
    const int lane = threadIdx.x & 31;
    constexpr int N = PER * 32;
    unsigned long long v[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) v[q] = q * 32 + lane < n ? list[q * 32 + lane] : 0ull;
#pragma unroll 1
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll 1
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 32) {
                const int qs = stride / 32;
#pragma unroll
                for (int q = 0; q < PER; ++q) {
#pragma unroll
                    for (int p2 = q + 1; p2 < PER; ++p2) {
                        if ((q ^ p2) != qs) continue;
                        const bool desc = ((q * 32 + lane) & size) == 0;
                        const unsigned long long a = v[q], b = v[p2];
                        const bool sw = desc ? (a < b) : (a > b);
                        v[q] = sw ? b : a;
                        v[p2] = sw ? a : b;
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    const int i = q * 32 + lane;
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[q], stride);
                    const bool keep_max = ((i & stride) == 0) == ((i & size) == 0);
                    v[q] = keep_max ? (v[q] > o ? v[q] : o) : (v[q] < o ? v[q] : o);
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < PER; ++q) list[q * 32 + lane] = v[q];
    __syncwarp();
}

__device__ __noinline__ void warp_sort_list(unsigned long long* list, int n)
{
    if (n <= 32) warp_sort_words<1>(list, n);
    else if (n <= 64) warp_sort_words<2>(list, n);
    else if (n <= 128) warp_sort_words<4>(list, n);
    else warp_sort_words<8>(list, n);
}

// Warp 0 of the leader: the same cut as resolve_cut, for short lists, with warp
// reductions and scans only.
__device__ __noinline__ void resolve_cut_warp(GShared& sh, const unsigned long long* list, int total, int f)
{
    const int lane = threadIdx.x & 31;
    const RowParams& rp = sh.rp[f];
    ForkOut& fo = sh.bc.f[f];
    const float m = sh.bc.m;
    const uint32_t tkey = f2key(fo.tau);
    int c = 0;
    for (int i = lane; i < total; i += 32) c += cand_key(list[i]) >= tkey ? 1 : 0;
    const int nf = __reduce_add_sync(0xffffffffu, c);
    const bool dom_complete = rp.do_topk && nf >= rp.k;
    const int dn = rp.do_topk ? min(rp.k, nf) : nf;
    bool unresolved = dn < 1;
    int np = dn;
    if (rp.do_topp && !unresolved) {
        const int per = (dn + 31) / 32;
        const int i0 = min(dn, lane * per), i1 = min(dn, i0 + per);
        float ls = 0.0f, lc = 0.0f;
        for (int i = i0; i < i1; ++i) {
            const float e = expf((key2f(cand_key(list[i])) - m) * rp.invT);
            const float y = e - lc;
            const float t = ls + y;
            lc = (t - ls) - y;
            ls = t;
        }
        const double loc = double(ls) - double(lc);
        double incl = loc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const double tot = __shfl_sync(0xffffffffu, incl, 31);
        double zdom = sh.zrow[f];
        if (rp.do_topk) {
            if (!dom_complete) unresolved = true;
            zdom = tot;
        }
        const double pz = double(rp.p) * zdom;
        int first = INT_MAX;
        double sacc = incl - loc;
        for (int i = i0; i < i1; ++i) {
            if (i > 0 && sacc >= pz) {
                first = i;
                break;
            }
            sacc += double(expf((key2f(cand_key(list[i])) - m) * rp.invT));
        }
        first = __reduce_min_sync(0xffffffffu, first);
        const bool minp_caps = rp.do_minp && fo.tau <= fo.xthr;
        if (first != INT_MAX) np = first;
        else if (!dom_complete && tot < pz && !minp_caps) unresolved = true;
    } else if (rp.do_topk && !dom_complete && !(rp.do_minp && fo.tau <= fo.xthr)) {
        unresolved = true;
    }
    if (unresolved) {
        if (lane == 0) fo.kind = kKindExact;
        __syncwarp();
        return;
    }
    int nk = np;
    if (rp.do_minp) {
        int b = INT_MAX;
        for (int i = lane; i < np; i += 32)
            if (key2f(cand_key(list[i])) < fo.xthr) b = min(b, i);
        b = __reduce_min_sync(0xffffffffu, b);
        nk = b == INT_MAX ? np : max(b, 1);
    }
    if (lane == 0) {
        const unsigned long long last = list[nk - 1];
        fo.bkey = cand_key(last);
        fo.bidx = cand_idx(last);
        fo.has_bound = 1;
        fo.kind = kKindPick;
        fo.listed = 1;
    }
    __syncwarp();
}

// Warp 0 of the leader: sort a short list and cut every listed fork from it;
// a fork whose parameters and bound match an earlier listed fork copies its cut.
__device__ __noinline__ void warp_cut_lists(GShared& sh, unsigned long long* list, int total, int g)
{
    const int lane = threadIdx.x & 31;
    warp_sort_list(list, total);
    for (int f = 0; f < g; ++f) {
        if (sh.bc.f[f].kind != kKindList) continue;
        const RowParams& rp = sh.rp[f];
        int twin = -1;
        for (int e = 0; e < f; ++e) {
            const RowParams& re = sh.rp[e];
            const ForkOut& fe = sh.bc.f[e];
            if (fe.kind == kKindPick && fe.listed && re.k == rp.k && re.p == rp.p && re.minp == rp.minp &&
                re.invT == rp.invT && re.do_topk == rp.do_topk && re.do_topp == rp.do_topp &&
                re.do_minp == rp.do_minp && fe.tau == sh.bc.f[f].tau && sh.zrow[e] == sh.zrow[f])
                twin = e;
        }
        if (twin < 0) {
            resolve_cut_warp(sh, list, total, f);
            continue;
        }
        if (lane == 0) {
            ForkOut& fo = sh.bc.f[f];
            const ForkOut& fe = sh.bc.f[twin];
            fo.kind = kKindPick;
            fo.listed = 1;
            fo.has_bound = fe.has_bound;
            fo.bkey = fe.bkey;
            fo.bidx = fe.bidx;
        }
        __syncwarp();
    }
}

}  // namespace grp
}  // namespace dst

namespace dst {
namespace grp {

// Exact path of fork f (every CTA of the cluster): radix selects by count (top-k)
// and by fixed-point softmax mass (top-p over the top-k domain) over the staged row.
// Leaves the fork's bound set and kind Pick.
template <typename InT>
__device__ __noinline__ void exact_fork(GShared& sh, Part pt, uint32_t rank, uint32_t C, int f)
{
    const RowParams rp = sh.rp[f];
    const float m = sh.bc.m;
    uint32_t bk = 0;
    int bi = 0;
    bool dom = false;
    if (rp.do_topk) {
        exact_select<InT>(sh, pt, rp, rank, C, false, false, 0u, 0, m, (unsigned long long)rp.k, bk, bi);
        dom = true;
    }
    if (rp.do_topp) {
        exact_select<InT>(sh, pt, rp, rank, C, true, dom, bk, bi, m, 0ull, bk, bi);
        dom = true;
    }
    // every CTA computed the same bound
    if (threadIdx.x == 0) {
        ForkOut& fo = sh.bc.f[f];
        fo.has_bound = dom ? 1 : 0;
        fo.bkey = bk;
        fo.bidx = bi;
        fo.kind = kKindPick;
    }
    __syncthreads();
}

// Gumbel-max over the whole part for an untruncated fork: the part's best two.
template <typename InT>
__device__ __noinline__ void plain_fork(GShared& sh, Part pt, int f)
{
    const RowParams rp = sh.rp[f];
    GumbelAcc g;
    gumbel_init(g);
    part_for_each<InT>(pt, rp, [&](int v, float x) { gumbel_visit(g, rp, v, x); });
    const GTop2 t = block_top2(g.t, sh);
    if (threadIdx.x == 0) sh.part.g[f] = t;
    __syncthreads();
}

// Pick pass of fork f over this CTA's part: the best two Gumbel scores among the
// kept tokens and their mass relative to the row max.
// One warp's pick pass of a listed fork f over this CTA's candidate list: the best
// two exact fp32 Gumbel scores among the kept tokens and their mass (lane 0 stores).
__device__ __noinline__ void pick_warp(GShared& sh, int f, const unsigned long long* cand, int ncand)
{
    const int lane = threadIdx.x & 31;
    const RowParams& rp = sh.rp[f];
    const ForkOut& fo = sh.bc.f[f];
    const float m = sh.bc.m;
    const bool hb = fo.has_bound != 0, mp = rp.do_minp != 0;
    const float a2 = rp.invT * 1.4426950408889634f;
    GTop2 t;
    t.a = grec_empty();
    t.b = grec_empty();
    float s = 0.0f, comp = 0.0f;
    for (int i = lane; i < ncand; i += 32) {
        const unsigned long long w = cand[i];
        const float x = key2f(cand_key(w));
        const int v = cand_idx(w);
        if (!(x > -INFINITY)) continue;
        if (hb && !in_prefix(cand_key(w), v, fo.bkey, fo.bidx)) continue;
        if (mp && !(x >= fo.xthr)) continue;
        if (!rp.greedy) {
            const uint32_t word = noise_word(rp, v);
            top2_insert(t, GRec{x * rp.invT - logf(noise_exp1_f32(word)), v, x, word});
        }
        if (rp.want_out) {
            const float e = exp2f((x - m) * a2);
            const float y = e - comp;
            const float u = s + y;
            comp = (u - s) - y;
            s = u;
        }
    }
    top2_warp_reduce(t);
    double z = double(s) - double(comp);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (lane == 0) {
        sh.part.g[f] = t;
        sh.part.zk[f] = z;
    }
}

// A fork whose kept tokens are all listed reads only this CTA's candidate list.
template <typename InT>
__device__ __noinline__ void pick_part(GShared& sh, Part pt, int f, const unsigned long long* cand,
                                       int ncand)
{
    const RowParams rp = sh.rp[f];
    const ForkOut fo = sh.bc.f[f];
    const float m = sh.bc.m;
    const bool hb = fo.has_bound != 0, mp = rp.do_minp != 0;
    const float a2 = rp.invT * 1.4426950408889634f;
    GumbelAcc g;
    gumbel_init(g);
    float s = 0.0f, comp = 0.0f;
    auto visit = [&](int v, float x) {
        if (!(x > -INFINITY)) return;
        if (hb && !in_prefix(f2key(x), v, fo.bkey, fo.bidx)) return;
        if (mp && !(x >= fo.xthr)) return;
        if (!rp.greedy) gumbel_visit(g, rp, v, x);
        if (rp.want_out) {
            const float e = exp2f((x - m) * a2);
            const float y = e - comp;
            const float t = s + y;
            comp = (t - s) - y;
            s = t;
        }
    };
    if (fo.listed) {
        for (int i = threadIdx.x; i < ncand; i += kT) {
            const unsigned long long w = cand[i];
            visit(cand_idx(w), key2f(cand_key(w)));
        }
    } else {
        part_for_each<InT>(pt, rp, visit);
    }
    const GTop2 t = block_top2(g.t, sh);
    const double z = block_sum_f64(double(s) - double(comp), sh);
    if (threadIdx.x == 0) {
        sh.part.g[f] = t;
        sh.part.zk[f] = z;
    }
    __syncthreads();
}

// fp32 probs / logprobs of fork f over this CTA's part: 16-byte streaming stores
// where the output row allows, plain stores for the ragged ends.
template <typename InT>
__device__ __noinline__ void write_outputs(const GShared& sh, const KernelParams& K, Part pt, int r, int f)
{
    const RowParams& rp = sh.rp[f];
    const ForkOut& fo = sh.bc.f[f];
    const int64_t base = int64_t(r) * K.vocab + pt.v0;
    float* op = K.out_probs ? K.out_probs + base : nullptr;
    float* ol = K.out_logprobs ? K.out_logprobs + base : nullptr;
    const bool bad = fo.status != kRowOk;
    const float m = sh.bc.m, lnz = fo.lnz, Te = rp.Te, xthr = fo.xthr;
    const bool hb = fo.has_bound != 0, mp = rp.do_minp != 0;
    const uint32_t bkey = fo.bkey;
    const int bidx = fo.bidx;
    auto val = [&](int i, float& pr, float& lp) {
        if (bad) {
            pr = lp = nan_f();
            return;
        }
        const float x = part_x<InT>(pt, rp, i);
        bool kept = x > -INFINITY;
        if (kept && hb) kept = in_prefix(f2key(x), pt.v0 + i, bkey, bidx);
        if (kept && mp) kept = x >= xthr;
        lp = -INFINITY;
        pr = 0.0f;
        if (kept) {
            lp = __fdiv_rn(x - m, Te) - lnz;
            pr = expf(lp);
        }
    };
    // the first element whose output address is 16-byte aligned (both outputs share it)
    const float* any = op ? op : ol;
    int head = int(((16u - (reinterpret_cast<uintptr_t>(any) & 15u)) & 15u) / 4u);
    if (op && ol && ((reinterpret_cast<uintptr_t>(op) ^ reinterpret_cast<uintptr_t>(ol)) & 15u)) head = pt.n;
    head = min(head, pt.n);
    const int nv = (pt.n - head) / 4;
    for (int i = threadIdx.x; i < head; i += kT) {
        float pr, lp;
        val(i, pr, lp);
        if (op) op[i] = pr;
        if (ol) ol[i] = lp;
    }
    for (int q = threadIdx.x; q < nv; q += kT) {
        const int i = head + 4 * q;
        float4 P4, L4;
        val(i, P4.x, L4.x);
        val(i + 1, P4.y, L4.y);
        val(i + 2, P4.z, L4.z);
        val(i + 3, P4.w, L4.w);
        if (op) __stcs(reinterpret_cast<float4*>(op + i), P4);
        if (ol) __stcs(reinterpret_cast<float4*>(ol + i), L4);
    }
    for (int i = head + 4 * nv + threadIdx.x; i < pt.n; i += kT) {
        float pr, lp;
        val(i, pr, lp);
        if (op) op[i] = pr;
        if (ol) ol[i] = lp;
    }
}

}  // namespace grp
}  // namespace dst

namespace dst {
namespace grp {

// Leader CTA: concatenate the C candidate lists (counts.n[c] words in CTA c) into
// `list`; each thread issues all its remote loads before storing any. The counts
// come by value and are indexed by constants only, so they stay in registers.
struct PartCounts {
    uint32_t n[kMaxParts];
};
__device__ __noinline__ void gather_lists(unsigned long long* list, const unsigned long long* cand,
                                          const PartCounts counts, uint32_t C, int total)
{
    constexpr int kU = 16;  // list capacity / kT
    const int tid = threadIdx.x;
    unsigned long long w[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int gi = tid + u * kT;
        w[u] = 0ull;
        if (gi < total) {
            int c = 0, li = gi;
#pragma unroll
            for (int cc = 0; cc + 1 < kMaxParts; ++cc) {
                if (c == cc && cc + 1 < int(C) && li >= int(counts.n[cc])) {
                    li -= int(counts.n[cc]);
                    c = cc + 1;
                }
            }
            w[u] = dsmem_ld_u64(dsmem_map(smem_addr(&cand[li]), uint32_t(c)));
        }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
        if (tid + u * kT < total) list[tid + u * kT] = w[u];
    __syncthreads();
}

template <typename InT, bool kPen>
__global__ void __launch_bounds__(kT, 2) group_kernel(const __grid_constant__ GroupParams P)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    GShared& sh = *reinterpret_cast<GShared*>(smem_raw);
    unsigned long long* list = reinterpret_cast<unsigned long long*>(smem_raw + P.off_list);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem_raw + P.off_cand);
    uint16_t* cnt = reinterpret_cast<uint16_t*>(smem_raw + P.off_cnt);
    unsigned char* stage = smem_raw + P.off_stage;
    constexpr int ES = int(sizeof(InT));
    const KernelParams& K = P.k;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint32_t rank = cluster_ctarank(), C = cluster_nctarank();
    const int V = int(K.vocab), L = P.slice_len;
    const int v0 = int(rank) * L;
    const int n = max(0, min(V - v0, L));
    const int ncl = int(gridDim.x / C);
    const int n_tmax = int(C) * kT;

    if (tid == 0) {
        for (int c = 0; c < kChunks; ++c) mbar_init(&sh.mbar[c], 1);
        fence_mbar_init();
    }
    uint32_t phase_bits = 0;  // parity of the next completion of each mbarrier
    uint32_t stuck_bits = 0;  // barriers whose copies never completed (the CTA stops copying)
    __syncthreads();

    // Chunks of output rows: a cluster's first one is its index; it claims each
    // next one from the work counter while it serves the current one (at the
    // end of the chunk's first group, when every CTA of the cluster is known to
    // run), so that clusters whose groups run long take fewer chunks. The claim
    // reaches every CTA through the cluster barrier that closes the group.
    int chunk = int(cluster_id_x());
    for (int it = 0; chunk < P.n_chunks; ++it) {
        bool claimed = false;
        const int cr0 = chunk * P.chunk, cr1 = min(P.n_rows, cr0 + P.chunk);
        for (int r0 = cr0; r0 < cr1;) {
            // ---- set-up (warp 0): the group, its bulk copies, its forks' parameters
            if (wid == 0) {
                const int lim = P.group ? min(kMaxForks, cr1 - r0) : 1;
                int lr = -1;
                if (lane < lim) lr = K.logit_row ? K.logit_row[r0 + lane] : r0 + lane;
                const int lr0 = __shfl_sync(0xffffffffu, lr, 0);
                const unsigned same = __ballot_sync(0xffffffffu, lane < lim && lr == lr0);
                const int g = __ffs(~same) - 1;
                const bool lrow_ok = lr0 >= 0 && int64_t(lr0) < K.n_logit_rows;
                if (lane == 0) {
                    int nch = 0, hb = 0, head_end = n, tail_begin = n;
                    if (lrow_ok && n > 0 && stuck_bits == 0) {
                        const unsigned char* gp = static_cast<const unsigned char*>(K.logits) +
                                                  (int64_t(lr0) * K.row_stride + v0) * ES;
                        const uintptr_t a = reinterpret_cast<uintptr_t>(gp);
                        hb = int(a & 15u);
                        const uintptr_t A0 = (a + 15u) & ~uintptr_t(15);
                        const uintptr_t A1 = (a + uintptr_t(n) * ES) & ~uintptr_t(15);
                        if (A1 > A0) {
                            head_end = int((A0 - a) / ES);
                            tail_begin = int((A1 - a) / ES);
                            const uint32_t bytes = uint32_t(A1 - A0);
                            const uint32_t per = ((bytes / kChunks) + 15u) & ~15u;
                            // order this CTA's earlier reads of the buffer before the copies
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            uint32_t done = 0;
                            while (done < bytes && nch < kChunks) {
                                const uint32_t b = min(per ? per : bytes, bytes - done);
                                mbar_arrive_expect_tx(&sh.mbar[nch], b);
                                bulk_copy_g2s(stage + (A0 - (a - hb)) + done,
                                              reinterpret_cast<const void*>(A0 + done), b, &sh.mbar[nch]);
                                done += b;
                                ++nch;
                            }
                        }
                    }
                    sh.nch = nch;
                    sh.hb = hb;
                    sh.head_end = head_end;
                    sh.tail_begin = tail_begin;
                    sh.n_forks = g;
                    sh.r0 = r0;
                    sh.lrow = lrow_ok ? lr0 : -1;
                }
                if (lane < g) {
                    read_row_params(K, r0 + lane, sh.rp[lane]);
                    if (!lrow_ok) sh.rp[lane].status = kRowBadParam;
                }
                __syncwarp();
                if (lane == 0) {
                    // forks that need the row's mass share it per temperature
                    int ns = 0;
                    for (int f = 0; f < g; ++f) {
                        sh.zslot_of[f] = -1;
                        if (!fork_needs_z(sh.rp[f], n_tmax)) continue;
                        int s = 0;
                        while (s < ns && sh.rp[sh.zslot_fork[s]].Te != sh.rp[f].Te) ++s;
                        if (s == ns) sh.zslot_fork[ns++] = f;
                        sh.zslot_of[f] = s;
                    }
                    sh.zslots = ns;
                }
            }
            if (wid == 1) {
                // Te * ln(min_p) per row, in double (a slow operation here: off the
                // leader's path, beside warp 0's loads)
                const int lim = P.group ? min(kMaxForks, cr1 - r0) : 1;
                if (lane < lim) {
                    const int r = r0 + lane;
                    const float mp = K.min_p ? K.min_p[r] : 0.0f;
                    const float T = K.temperature[r];
                    const double Te = T < 1e-5f ? 1.0 : double(T);
                    sh.lnmp[lane] = (mp > 0.0f && mp <= 1.0f) ? Te * log(double(mp)) : 0.0;
                }
            }
            __syncthreads();
            const int g = sh.n_forks;
            const bool row_ok = sh.lrow >= 0;
            const RowParams& rp0 = sh.rp[0];
            Part pt;
            pt.stage = stage;
            pt.cnt = nullptr;
            pt.n = n;
            pt.hoff = sh.hb / ES;
            pt.v0 = v0;

            // head / tail elements outside the 16-byte-aligned interior: plain loads
            if (row_ok && n > 0) {
                const unsigned char* gp = static_cast<const unsigned char*>(K.logits) +
                                          (int64_t(sh.lrow) * K.row_stride + v0) * ES;
                const int hend = sh.head_end, tbeg = sh.tail_begin, hb = sh.hb;
                for (int i = tid; i < hend; i += kT) {
                    if (ES == 4) reinterpret_cast<float*>(stage + hb)[i] = reinterpret_cast<const float*>(gp)[i];
                    else reinterpret_cast<uint16_t*>(stage + hb)[i] = reinterpret_cast<const uint16_t*>(gp)[i];
                }
                for (int i = tbeg + tid; i < n; i += kT) {
                    if (ES == 4) reinterpret_cast<float*>(stage + hb)[i] = reinterpret_cast<const float*>(gp)[i];
                    else reinterpret_cast<uint16_t*>(stage + hb)[i] = reinterpret_cast<const uint16_t*>(gp)[i];
                }
            }

            // history counts of this part (penalties; such groups hold one row)
            bool bad_hist = false;
            const bool pen = kPen && rp0.has_hist && rp0.status == kRowOk;
            if (pen) {
                uint4* c4 = reinterpret_cast<uint4*>(cnt);
                const int nw4 = (L * 2 + 15) / 16;
                for (int i = tid; i < nw4; i += kT) c4[i] = make_uint4(0, 0, 0, 0);
                __syncthreads();
                const int len = rp0.hhi - rp0.hlo;
                if (rp0.hlo < 0 || len < 0 || len > 65535) {
                    bad_hist = true;
                } else {
                    uint32_t* c32 = reinterpret_cast<uint32_t*>(cnt);
                    for (int j = rp0.hlo + tid; j < rp0.hhi; j += 4 * kT) {
                        int ids[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) ids[u] = j + u * kT < rp0.hhi ? K.hist_ids[j + u * kT] : 0;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (j + u * kT >= rp0.hhi) continue;
                            const int id = ids[u];
                            if (id < 0 || id >= V) bad_hist = true;
                            else if (id >= v0 && id < v0 + n) {
                                const int i = id - v0;
                                atomicAdd(&c32[i >> 1], 1u << (16 * (i & 1)));
                            }
                        }
                    }
                }
            }
            bad_hist = __syncthreads_or(bad_hist);

            // wait for the bulk copies (bounded)
            bool timeout = stuck_bits != 0 && row_ok && n > 0;
            const int nch = sh.nch;
            uint32_t tb = 0;
            for (int c = 0; c < nch; ++c)
                if (!mbar_wait_bounded(&sh.mbar[c], (phase_bits >> c) & 1u, kPolls)) tb |= 1u << c;
            phase_bits ^= (1u << nch) - 1u;
            tb = __syncthreads_or(tb != 0) ? ((1u << nch) - 1u) : 0u;
            stuck_bits |= tb;
            timeout = __syncthreads_or(timeout || tb != 0);

            if (pen && !bad_hist) {
                if (ES == 4) {
                    // fp32 rows: penalise in place once per distinct history token; the
                    // thread that clears a token's count applies its penalty
                    float* xs = reinterpret_cast<float*>(stage + sh.hb);
                    uint32_t* c32 = reinterpret_cast<uint32_t*>(cnt);
                    for (int j = rp0.hlo + tid; j < rp0.hhi; j += kT) {
                        const int id = K.hist_ids[j];
                        if (id < v0 || id >= v0 + n) continue;
                        const int i = id - v0;
                        const int sft = 16 * (i & 1);
                        const uint32_t old = atomicAnd(&c32[i >> 1], ~(0xFFFFu << sft));
                        const uint32_t c = (old >> sft) & 0xFFFFu;
                        if (c) xs[i] = penalize(xs[i], c, rp0);
                    }
                    __syncthreads();
                } else {
                    pt.cnt = cnt;
                }
            }

            // ---- P1: max / argmax / flags and thread maxima
            const bool base_ok = row_ok && !timeout && !bad_hist;
            {
                float mx = -INFINITY;
                int am = INT_MAX;
                bool nonfin = false, anyfin = false;
                if (base_ok && pt.cnt == nullptr) {
                    // whole vectors: their maximum first, the position only when it improves
                    constexpr int EPV = VecMax<InT>::E;
                    const uint4* vec = reinterpret_cast<const uint4*>(stage);
                    const int j_lo = (pt.hoff + EPV - 1) / EPV, j_hi = (pt.hoff + n) / EPV;
                    for (int j = j_lo + tid; j < j_hi; j += kT) {
                        const uint4 raw = vec[j];
                        bool vn;
                        const float vm = VecMax<InT>::vmax(raw, vn);
                        nonfin |= vn || vm == INFINITY;
                        anyfin |= vm > -INFINITY && vm < INFINITY;
                        if (vm > mx) {
                            mx = vm;
                            am = v0 + j * EPV - pt.hoff + vec_first<InT>(raw, vm);
                        }
                    }
                    // the ragged ends, element by element
                    auto one = [&](int i) {
                        const float x = part_x<InT>(pt, rp0, i);
                        if (x != x || x == INFINITY) nonfin = true;
                        else if (x > -INFINITY) anyfin = true;
                        if (x > mx || (x == mx && v0 + i < am)) {
                            mx = x;
                            am = v0 + i;
                        }
                    };
                    const int head = min(n, j_lo * EPV - pt.hoff);
                    const int tail = max(head, j_hi * EPV - pt.hoff);
                    for (int i = tid; i < head; i += kT) one(i);
                    for (int i = tail + tid; i < n; i += kT) one(i);
                } else if (base_ok) {
                    part_for_each<InT>(pt, rp0, [&](int v, float x) {
                        if (x != x || x == INFINITY) nonfin = true;
                        else if (x > -INFINITY) anyfin = true;
                        if (x > mx) {
                            mx = x;
                            am = v;
                        }
                    });
                }
                sh.tmax[tid] = f2key(mx);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float om = __shfl_xor_sync(0xffffffffu, mx, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, am, off);
                    maxidx_merge(mx, am, om, oi);
                }
                const bool wnf = __any_sync(0xffffffffu, nonfin), waf = __any_sync(0xffffffffu, anyfin);
                if (lane == 0) {
                    sh.red_f[wid] = mx;
                    sh.red_i[wid] = am;
                    sh.red_u[wid] = (wnf ? kFlagNonFinite : 0u) | (waf ? kFlagAnyFinite : 0u);
                }
                __syncthreads();
                if (tid == 0) {
                    float m = -INFINITY;
                    int a = INT_MAX;
                    uint32_t fl = (bad_hist ? kFlagBadHistory : 0u) | (timeout ? kFlagTimeout : 0u);
                    for (int w = 0; w < kW; ++w) {
                        maxidx_merge(m, a, sh.red_f[w], sh.red_i[w]);
                        fl |= sh.red_u[w];
                    }
                    sh.part.mx = m;
                    sh.part.amax = a;
                    sh.part.flags = fl;
                }
                __syncthreads();
            }
            const float mc = sh.part.mx;
            const bool part_fin = base_ok && mc > -INFINITY && mc < INFINITY;
            // the part's softmax mass per temperature slot
            for (int s = 0; s < sh.zslots; ++s) {
                double z = 0.0;
                if (part_fin) z = part_mass<InT>(pt, sh.rp[sh.zslot_fork[s]], mc, sh);
                if (tid == 0) sh.part.z[s] = z;
            }
            // Gumbel-max of the forks that truncate nothing
            for (int f = 0; f < g; ++f) {
                const RowParams& rp = sh.rp[f];
                if (rp.status != kRowOk || rp.greedy || fork_truncates(rp)) continue;
                if (base_ok) {
                    plain_fork<InT>(sh, pt, f);
                } else if (tid == 0) {
                    sh.part.g[f].a = grec_empty();
                    sh.part.g[f].b = grec_empty();
                }
            }
            __syncthreads();
            cluster_sync();

            // ---- R1 (leader): row max, status, early picks, bounds of the kept sets
            if (rank == 0) {
                if (wid == 0) {
                    const bool have = lane < int(C);
                    float qm = -INFINITY;
                    int qa = INT_MAX;
                    uint32_t qf = 0;
                    if (have) {
                        qm = dsmem_ld_f32(dsmem_map(smem_addr(&sh.part.mx), uint32_t(lane)));
                        qa = int(dsmem_ld_u32(dsmem_map(smem_addr(&sh.part.amax), uint32_t(lane))));
                        qf = dsmem_ld_u32(dsmem_map(smem_addr(&sh.part.flags), uint32_t(lane)));
                    }
                    float m = qm;
                    int a = qa;
                    uint32_t fl = qf;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const float om = __shfl_xor_sync(0xffffffffu, m, off);
                        const int oi = __shfl_xor_sync(0xffffffffu, a, off);
                        maxidx_merge(m, a, om, oi);
                        fl |= __shfl_xor_sync(0xffffffffu, fl, off);
                    }
                    // the row's mass per slot, rescaled from each part's max to m
                    for (int s = 0; s < sh.zslots; ++s) {
                        double z = 0.0;
                        if (have && qm > -INFINITY && m < INFINITY) {
                            const double zc = __longlong_as_double(
                                (long long)dsmem_ld_u64(dsmem_map(smem_addr(&sh.part.z[s]), uint32_t(lane))));
                            z = zc * double(expf((qm - m) * sh.rp[sh.zslot_fork[s]].invT));
                        }
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
                        if (lane == 0)
                            for (int f = 0; f < g; ++f)
                                if (sh.zslot_of[f] == s) sh.zrow[f] = z;
                    }
                    // plain forks: the best two of the parts (kept in the leader's own partial)
                    for (int f = 0; f < g; ++f) {
                        const RowParams& rp = sh.rp[f];
                        if (rp.status != kRowOk || rp.greedy || fork_truncates(rp)) continue;
                        GTop2 t;
                        t.a = grec_empty();
                        t.b = grec_empty();
                        if (have) dsmem_read(t, sh.part.g[f], uint32_t(lane));
                        top2_warp_reduce(t);
                        __syncwarp();
                        if (lane == 0) sh.part.g[f] = t;
                    }
                    __syncwarp();
                    // one lane per fork: status, kind, min-p threshold, early token
                    if (lane < g) {
                        const int f = lane;
                        const RowParams& rp = sh.rp[f];
                        ForkOut fo;
                        fo.status = rp.status;
                        if (fo.status == kRowOk) {
                            if (fl & kFlagBadHistory) fo.status = kRowBadHistory;
                            else if (fl & kFlagTimeout) fo.status = kRowTimeout;
                            else if (fl & kFlagNonFinite) fo.status = kRowNonFinite;
                            else if (!(fl & kFlagAnyFinite)) fo.status = kRowAllNegInf;
                        }
                        fo.token = -1;
                        fo.kind = kKindDone;
                        fo.has_bound = 0;
                        fo.xthr = -INFINITY;
                        fo.tau = -INFINITY;
                        fo.lnz = 0.0f;
                        fo.bkey = 0;
                        fo.bidx = 0;
                        fo.listed = 0;
                        if (fo.status == kRowOk) {
                            const bool trunc = fork_truncates(rp);
                            if (rp.greedy) fo.token = a;
                            else if (!trunc) fo.token = settle_pair(sh.part.g[f], rp.T);
                            if (rp.do_minp) {
                                const double th = double(m) + sh.lnmp[f];
                                float x = float(th);
                                if (double(x) < th) x = nextafterf(x, INFINITY);
                                fo.xthr = x;
                            }
                            if (!trunc) {
                                if (rp.want_out) {
                                    fo.kind = kKindAll;
                                    fo.lnz = logf(float(sh.zrow[f]));
                                }
                            } else if (rp.want_out || !rp.greedy) {
                                // min-p alone: the kept set is every token >= the threshold,
                                // all of them in the candidate lists gathered at that bound
                                fo.kind = (rp.do_topk || rp.do_topp) ? kKindList : kKindPick;
                                if (fo.kind == kKindPick) {
                                    fo.tau = fo.xthr;
                                    fo.listed = 1;
                                }
                            }
                        }
                        sh.bc.f[f] = fo;
                    }
                    if (lane == 0) {
                        sh.bc.m = m;
                        sh.bc.amax = a;
                        sh.bc.status = 0;
                    }
                }
                __syncthreads();
                bool need_bounds = false;
                for (int f = 0; f < g; ++f) need_bounds |= sh.bc.f[f].kind == kKindList;
                __shared__ float s_tk[kMaxForks], s_tp[kMaxForks];
                if (need_bounds) tmax_bounds(sh, C, g, sh.bc.m, reinterpret_cast<uint32_t*>(list), s_tk, s_tp);
                if (tid == 0) {
                    float tau_all = INFINITY;
                    int gather = 0, exact = 0;
                    for (int f = 0; f < g; ++f) {
                        ForkOut& fo = sh.bc.f[f];
                        if (fo.kind == kKindPick && fo.listed) {
                            tau_all = fminf(tau_all, fo.tau);
                            gather = 1;
                        }
                        if (fo.kind != kKindList) continue;
                        const RowParams& rp = sh.rp[f];
                        const bool want_k = rp.do_topk && rp.k <= n_tmax;
                        const bool have_k = want_k && s_tk[f] == s_tk[f];
                        const bool have_p = !want_k && rp.do_topp && s_tp[f] == s_tp[f];
                        float tau = -INFINITY;
                        bool bounded;
                        if (want_k) {
                            // the list must hold the whole top-k set when top-p cuts inside it;
                            // otherwise min-p may raise the bound
                            bounded = have_k || (rp.do_minp && !rp.do_topp);
                            if (have_k) tau = s_tk[f];
                            if (rp.do_minp && !rp.do_topp) tau = fmaxf(tau, fo.xthr);
                        } else if (rp.do_topp) {
                            bounded = have_p;
                            if (have_p) tau = s_tp[f];
                            if (rp.do_minp) tau = fmaxf(tau, fo.xthr);
                        } else {
                            // top-k above the thread-maxima count: min-p alone can bound it
                            bounded = rp.do_minp;
                            tau = fo.xthr;
                        }
                        if (bounded && tau > -INFINITY) {
                            fo.tau = tau;
                            tau_all = fminf(tau_all, tau);
                            gather = 1;
                        } else {
                            fo.kind = kKindExact;
                            exact = 1;
                        }
                    }
                    sh.bc.tau_all = tau_all;
                    sh.bc.gather = gather;
                    sh.bc.exact = exact;
                    sh.bc.out = K.out_probs != nullptr || K.out_logprobs != nullptr;
                }
                __syncthreads();
                bcast_cluster(sh.bc, C);
            }
            cluster_sync();

            // ---- P2: every token at or above the smallest bound; R2 (leader): the cuts
            if (sh.bc.gather) {
                if (tid == 0) sh.ncand = 0;
                __syncthreads();
                const float tau = sh.bc.tau_all;
                const int cap = P.part_cap;
                auto add = [&](int v, float x) {
                    if (x >= tau) {
                        const int pos = atomicAdd(&sh.ncand, 1);
                        if (pos < cap) cand[pos] = cand_word(f2key(x), v);
                    }
                };
                if (pt.cnt == nullptr) {
                    // whole vectors: skip those whose maximum is below the bound
                    constexpr int EPV = VecMax<InT>::E;
                    const uint4* vec = reinterpret_cast<const uint4*>(stage);
                    const int j_lo = (pt.hoff + EPV - 1) / EPV, j_hi = (pt.hoff + n) / EPV;
                    for (int j = j_lo + tid; j < j_hi; j += kT) {
                        const uint4 raw = vec[j];
                        bool vn;
                        if (!(VecMax<InT>::vmax(raw, vn) >= tau)) continue;
#pragma unroll
                        for (int e = 0; e < EPV; ++e) add(v0 + j * EPV + e - pt.hoff, ElemTraits<InT>::get(raw, e));
                    }
                    const int head = min(n, j_lo * EPV - pt.hoff);
                    const int tail = max(head, j_hi * EPV - pt.hoff);
                    for (int i = tid; i < head; i += kT) add(v0 + i, part_x<InT>(pt, rp0, i));
                    for (int i = tail + tid; i < n; i += kT) add(v0 + i, part_x<InT>(pt, rp0, i));
                } else {
                    part_for_each<InT>(pt, rp0, add);
                }
                __syncthreads();
                if (tid == 0) sh.part.ncand = uint32_t(sh.ncand);
                __syncthreads();
                cluster_sync();
                if (rank == 0) {
                    PartCounts counts;
                    uint32_t total = 0;
                    bool overflow = false;
#pragma unroll
                    for (int c = 0; c < kMaxParts; ++c)
                        counts.n[c] = c < int(C) ? dsmem_ld_u32(dsmem_map(smem_addr(&sh.part.ncand), uint32_t(c))) : 0u;
#pragma unroll
                    for (int c = 0; c < kMaxParts; ++c) {
                        overflow |= counts.n[c] > uint32_t(cap);
                        total += counts.n[c];
                    }
                    overflow |= total > uint32_t(P.list_cap);
                    bool need_sort = false;
                    for (int f = 0; f < g; ++f) need_sort |= sh.bc.f[f].kind == kKindList;
                    // short lists: warp 0 sorts and cuts alone (no block-wide waits)
                    const bool small = !overflow && need_sort && total <= 256u;
                    if (small) {
                        gather_lists(list, cand, counts, C, int(total));
                        if (wid == 0) warp_cut_lists(sh, list, int(total), g);
                        __syncthreads();
                    } else if (!overflow && need_sort) {
                        gather_lists(list, cand, counts, C, int(total));
                        sort_desc<unsigned long long>(list, int(total));
                    }
                    if (overflow) {
                        __syncthreads();
                        if (tid < g && sh.bc.f[tid].kind == kKindPick && sh.bc.f[tid].listed) sh.bc.f[tid].listed = 0;
                        __syncthreads();
                    }
                    for (int f = 0; f < g && !small; ++f) {
                        if (sh.bc.f[f].kind != kKindList) continue;
                        if (overflow) {
                            __syncthreads();
                            if (tid == 0) sh.bc.f[f].kind = kKindExact;
                            __syncthreads();
                            continue;
                        }
                        // forks with the same cut parameters share the cut
                        int twin = -1;
                        const RowParams& rp = sh.rp[f];
                        for (int e = 0; e < f; ++e) {
                            const RowParams& re = sh.rp[e];
                            const ForkOut& fe = sh.bc.f[e];
                            if (fe.kind == kKindPick && fe.listed && re.k == rp.k && re.p == rp.p &&
                                re.minp == rp.minp && re.invT == rp.invT && re.do_topk == rp.do_topk &&
                                re.do_topp == rp.do_topp && re.do_minp == rp.do_minp && fe.tau == sh.bc.f[f].tau &&
                                sh.zrow[e] == sh.zrow[f])
                                twin = e;
                        }
                        __syncthreads();
                        if (twin >= 0) {
                            if (tid == 0) {
                                ForkOut& fo = sh.bc.f[f];
                                const ForkOut& fe = sh.bc.f[twin];
                                fo.kind = kKindPick;
                                fo.listed = 1;
                                fo.has_bound = fe.has_bound;
                                fo.bkey = fe.bkey;
                                fo.bidx = fe.bidx;
                            }
                            __syncthreads();
                            continue;
                        }
                        resolve_cut(sh, list, int(total), f);
                    }
                    __syncthreads();
                    if (tid == 0) {
                        int exact = 0;
                        for (int f = 0; f < g; ++f) exact |= sh.bc.f[f].kind == kKindExact;
                        sh.bc.exact = exact;
                    }
                    __syncthreads();
                    bcast_cluster(sh.bc, C);
                }
                cluster_sync();
            }

            // ---- forks the list could not settle: exact path over the staged row
            if (sh.bc.exact) {
                for (int f = 0; f < g; ++f)
                    if (sh.bc.f[f].kind == kKindExact) exact_fork<InT>(sh, pt, rank, C, f);
            }

            // ---- pick pass: Gumbel-max and kept mass over the kept tokens of each fork;
            // a listed fork takes one warp over this CTA's candidates (all such forks at
            // once), any other the whole CTA over the staged part
            bool any_pick = false;
            for (int f = 0; f < g; ++f) {
                const RowParams& rp = sh.rp[f];
                const bool pk = sh.bc.f[f].kind == kKindPick && (!rp.greedy || rp.want_out);
                any_pick |= pk;
                if (pk && !sh.bc.f[f].listed) pick_part<InT>(sh, pt, f, cand, 0);
            }
            if (wid < g) {
                const RowParams& rp = sh.rp[wid];
                const ForkOut& fo = sh.bc.f[wid];
                if (fo.kind == kKindPick && fo.listed && (!rp.greedy || rp.want_out))
                    pick_warp(sh, wid, cand, min(sh.ncand, P.part_cap));
            }
            if (any_pick) {
                __syncthreads();
                cluster_sync();
                // leader: warp f merges fork f over the CTAs and settles it
                if (rank == 0 && wid < g) {
                    const int f = wid;
                    const RowParams& rp = sh.rp[f];
                    ForkOut& fo = sh.bc.f[f];
                    if (fo.kind == kKindPick && (!rp.greedy || rp.want_out)) {
                        const bool have = lane < int(C);
                        GTop2 t;
                        t.a = grec_empty();
                        t.b = grec_empty();
                        double z = 0.0;
                        if (have) {
                            dsmem_read(t, sh.part.g[f], uint32_t(lane));
                            z = __longlong_as_double(
                                (long long)dsmem_ld_u64(dsmem_map(smem_addr(&sh.part.zk[f]), uint32_t(lane))));
                        }
                        top2_warp_reduce(t);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
                        if (lane == 0) {
                            if (!rp.greedy) fo.token = settle_pair(t, rp.T);
                            if (rp.want_out) fo.lnz = logf(float(z));
                        }
                    }
                }
                __syncthreads();
                if (rank == 0 && sh.bc.out) bcast_cluster(sh.bc, C);
                cluster_sync();
            }

            // ---- P3: probs / logprobs
            if (sh.bc.out) {
                for (int f = 0; f < g; ++f) write_outputs<InT>(sh, K, pt, r0 + f, f);
            }
            if (rank == 0 && tid < g) {
                K.out_tokens[r0 + tid] = sh.bc.f[tid].token;
                if (K.out_status) K.out_status[r0 + tid] = sh.bc.f[tid].status;
            }
            if (!claimed && rank == 0 && tid == 0) {
                const int nx = ncl + int(atomicAdd(P.work, 1u));
                for (uint32_t c = 0; c < C; ++c)
                    dsmem_st_u32(dsmem_map(smem_addr(&sh.next_chunk[it & 1]), c), uint32_t(nx));
            }
            claimed = true;
            __syncthreads();
            cluster_sync();
            r0 += g;
        }
        chunk = sh.next_chunk[it & 1];
    }
    // the last cluster out clears the work counter for the next launch (every
    // cluster's claims come before its count)
    if (rank == 0 && tid == 0) {
        __threadfence();
        if (atomicAdd(P.work + 1, 1u) == uint32_t(ncl - 1)) {
            atomicExch(P.work, 0u);
            atomicExch(P.work + 1, 0u);
        }
    }
    // copies that gave up: wait (bounded) for them to land before the CTA exits
    for (int c = 0; c < kChunks; ++c)
        if (stuck_bits & (1u << c)) mbar_wait_bounded(&sh.mbar[c], ((phase_bits >> c) & 1u) ^ 1u, kPolls);
}

}  // namespace grp
}  // namespace dst
