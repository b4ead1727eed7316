// colsplit_kernel.cuh -- body of the column-split kernel (design in colsplit.cuh).
#pragma once

#include "colsplit.cuh"

namespace dst {
namespace col {

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Read the parameters of row r, validate them and classify the row.
__device__ __forceinline__ void load_row_info(const ColParams& P, int r, int lrow, bool lrow_ok,
                                              RowInfo& ri)
{
    const KernelParams& kp = P.k;
    const int64_t V = kp.vocab;
    ri.T = kp.temperature[r];
    ri.k = kp.top_k ? kp.top_k[r] : -1;
    ri.p = kp.top_p ? kp.top_p[r] : 1.0f;
    ri.minp = kp.min_p ? kp.min_p[r] : 0.0f;
    const bool seeded = kp.has_seed ? (kp.has_seed[r] != 0) : false;
    const uint64_t key = seeded ? kp.seed[r] : kp.global_seed;
    const uint32_t sid = kp.stream_id ? kp.stream_id[r] : (seeded ? 0u : uint32_t(r));
    ri.stream = (sid & 0x7FFFFFFFu) | (seeded ? 0x80000000u : 0u);
    ri.key_lo = uint32_t(key);
    ri.key_hi = uint32_t(key >> 32);
    const uint64_t off = kp.philox_offset_dev ? *kp.philox_offset_dev : kp.philox_offset;
    ri.off_lo = uint32_t(off);
    ri.off_hi = uint32_t(off >> 32);
    ri.lrow = lrow;
    bool bad = !lrow_ok;
    if (!(ri.T >= 0.0f) || isinf(ri.T)) bad = true;
    if (!(ri.k == -1 || ri.k >= 1)) bad = true;
    if (!(ri.p > 0.0f && ri.p <= 1.0f)) bad = true;
    if (!(ri.minp >= 0.0f && ri.minp <= 1.0f)) bad = true;
    if (kp.presence && !isfinite(kp.presence[r])) bad = true;
    if (kp.frequency && !isfinite(kp.frequency[r])) bad = true;
    if (kp.repetition && (!(kp.repetition[r] > 0.0f) || isinf(kp.repetition[r]))) bad = true;
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
}

template <typename InT>
struct SliceView {
    const unsigned char* st;
    int hoff, n, v0;
    __device__ __forceinline__ int nvec() const
    {
        constexpr int EPV = ElemTraits<InT>::kPerVec;
        return (hoff + n + EPV - 1) / EPV;
    }
};

// Phase A of one row on this CTA's slice, by one warp. Writes the record.
template <typename InT>
__device__ void slice_summary(const ColParams& P, ColShared& sh, int r, const SliceView<InT>& sv,
                              ColRec* rec)
{
    constexpr int EPV = ElemTraits<InT>::kPerVec;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const RowInfo& ri = sh.info[r];
    const uint8_t cls = ri.cls;
    const bool timeout = !mbar_wait_bounded(&sh.mbar[r], 0, kMaxPolls);
    const uint4* vec = reinterpret_cast<const uint4*>(sv.st);
    const int nvec = sv.nvec();
    float mx = -INFINITY;
    int am = INT_MAX;
    bool nonfin = false, anyfin = false;

    if (cls == kClsPlain) {
        const RowParams rp = as_row_params(ri);
        GumbelAcc g;
        gumbel_init(g);
        const float a2 = ri.invT * 1.4426950408889634f;  // log2 e / T
        for (int j = lane; j < nvec; j += 32) {
            const uint4 raw = vec[j];
            const int vb = sv.v0 + j * EPV - sv.hoff;  // token of element e = 0
            // the Philox blocks this vector touches, computed together (ILP)
            const uint32_t b0 = uint32_t(max(vb, 0)) >> 2;  // valid tokens are >= 0
            const uint4 k0 = philox4x32_10(make_uint4(b0, rp.stream, rp.off_lo, rp.off_hi),
                                           PhiloxKey{rp.key_lo, rp.key_hi});
            uint4 k1 = k0, k2 = k0;
            if (EPV > 4 || (vb & 3))
                k1 = philox4x32_10(make_uint4(b0 + 1, rp.stream, rp.off_lo, rp.off_hi),
                                   PhiloxKey{rp.key_lo, rp.key_hi});
            if (EPV > 4 && (vb & 3))
                k2 = philox4x32_10(make_uint4(b0 + 2, rp.stream, rp.off_lo, rp.off_hi),
                                   PhiloxKey{rp.key_lo, rp.key_hi});
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const int i = j * EPV + e - sv.hoff;
                if (i < 0 || i >= sv.n) continue;
                const float x = ElemTraits<InT>::get(raw, e);
                const int v = vb + e;
                if (x != x || x == INFINITY) nonfin = true;
                else if (x > -INFINITY) anyfin = true;
                if (x > mx) {
                    mx = x;
                    am = v;
                }
                if (!(x > -INFINITY)) continue;
                const uint32_t rel = (uint32_t(v) >> 2) - b0;
                const uint4 blk = rel == 0 ? k0 : (rel == 1 ? k1 : k2);
                const uint32_t w = lane_of(blk, uint32_t(v) & 3u);
                // score <= x/T - ln(1 - u); skip when that bound is below the entry bar
                if (fmaf(x, a2, -g.thr * 1.4426950408889634f) < __log2f(noise_one_minus_u(w))) continue;
                const float s = x * ri.invT - logf(noise_exp1_f32(w));
                const GRec rr{s, v, x, w};
                if (grec_better(rr, g.t.b)) {
                    top2_insert(g.t, rr);
                    const float s2 = g.t.b.s;
                    g.thr = s2 - (1e-4f + 1e-6f * fabsf(s2));
                }
            }
        }
        top2_warp_reduce(g.t);
        if (lane == 0) {
            rec->g0 = g.t.a;
            rec->g1 = g.t.b;
        }
    } else if (cls != kClsErr) {
        for (int j = lane; j < nvec; j += 32) {
            const uint4 raw = vec[j];
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const int i = j * EPV + e - sv.hoff;
                if (i < 0 || i >= sv.n) continue;
                const float x = ElemTraits<InT>::get(raw, e);
                if (x != x || x == INFINITY) nonfin = true;
                else if (x > -INFINITY) anyfin = true;
                if (x > mx) {
                    mx = x;
                    am = sv.v0 + i;
                }
            }
        }
    }
    const float lane_max = mx;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, off);
        const int oi = __shfl_xor_sync(0xffffffffu, am, off);
        maxidx_merge(mx, am, om, oi);
    }
    nonfin = __any_sync(0xffffffffu, nonfin);
    anyfin = __any_sync(0xffffffffu, anyfin);

    uint32_t nc = 0;
    if (cls == kClsCand) {
        // tau: the 8th largest lane maximum bounds the slice's 8th largest from below
        int rk = 0;
        for (int l = 0; l < 32; ++l) {
            const float o = __shfl_sync(0xffffffffu, lane_max, l);
            rk += (o > lane_max) || (o == lane_max && l < lane);
        }
        const unsigned bal = __ballot_sync(0xffffffffu, rk == kSliceCand - 1);
        const float tau = __shfl_sync(0xffffffffu, lane_max, bal ? __ffs(bal) - 1 : 0);
        unsigned long long* buf = sh.buf[wid];
        int cnt = 0;
        float zs = 0.0f, zc = 0.0f;  // compensated sum of exp((x - mx) / T)
        for (int j = lane; j - lane < nvec; j += 32) {
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (j < nvec) raw = vec[j];
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const int i = j * EPV + e - sv.hoff;
                const bool valid = j < nvec && i >= 0 && i < sv.n;
                const float x = ElemTraits<InT>::get(raw, e);
                const bool take = valid && x >= tau;
                const unsigned bt = __ballot_sync(0xffffffffu, take);
                if (take) {
                    const int pos = cnt + __popc(bt & ((1u << lane) - 1u));
                    if (pos < 64) buf[pos] = comp_of(x, sv.v0 + i);
                }
                cnt += __popc(bt);
                if (ri.need_z && valid && x > -INFINITY) {
                    const float t = __expf((x - mx) * ri.invT) - zc;
                    const float s2 = zs + t;
                    zc = (s2 - zs) - t;
                    zs = s2;
                }
            }
        }
        __syncwarp();
        if (cnt > 64) {
            nc = kOverflow;
        } else {
            unsigned long long a = lane < cnt ? buf[lane] : 0ull;
            unsigned long long b = lane + 32 < cnt ? buf[lane + 32] : 0ull;
            warp_sort64_desc(a, b);
            nc = uint32_t(min(cnt, kSliceCand));
            if (lane < kSliceCand) rec->cand[lane] = lane < int(nc) ? a : 0ull;
        }
        if (ri.need_z) {
            // combine the lanes' compensated sums (pairwise, fp32)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float os = __shfl_xor_sync(0xffffffffu, zs, off);
                const float oc = __shfl_xor_sync(0xffffffffu, zc, off);
                const float t = os - oc - zc;
                const float s2 = zs + t;
                zc = (s2 - zs) - t;
                zs = s2;
            }
            if (lane == 0) {
                rec->zs = zs;
                rec->zc = zc;
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        rec->mx = mx;
        rec->amax = am;
        rec->flags = (nonfin ? kFlagNonFinite : 0u) | (anyfin ? kFlagAnyFinite : 0u) |
                     (timeout ? kFlagTimeout : 0u);
        rec->nc = nc;
    }
}

// Finish row r from its records (one warp). Returns true when the row needs the
// CTA-wide exact path; m and amax are returned for it.
template <typename InT>
__device__ bool finish_row(const ColParams& P, ColShared& sh, int r, float& m_out, int& amax_out)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const KernelParams& kp = P.k;
    const RowInfo& ri = sh.info[r];
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
        if (fl & kFlagTimeout) status = kRowTimeout;
        else if (fl & kFlagNonFinite) status = kRowNonFinite;
        else if (!(fl & kFlagAnyFinite)) status = kRowAllNegInf;
    }
    m_out = m;
    amax_out = am;
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
        token = settle_top2(t, ri.T);
    } else {
        // ---- truncated row: merge the slices' candidates
        const bool small_k = ri.small_k;
        if (ri.do_topk && !small_k) fallback = true;
        unsigned long long tau_inc = 0ull;  // below this the merged list may miss tokens
        bool overflow = false;
        for (int s = lane; s < G; s += 32) {
            const uint32_t nc = __ldcg(&rr[s].nc);
            if (nc == kOverflow) overflow = true;
            else if (nc == uint32_t(kSliceCand)) {
                const unsigned long long c7 = __ldcg(&rr[s].cand[kSliceCand - 1]);
                tau_inc = c7 > tau_inc ? c7 : tau_inc;
            }
        }
        overflow = __any_sync(0xffffffffu, overflow);
        tau_inc = warp_max_u64(tau_inc);
        fallback = fallback || overflow;
        unsigned long long* buf = sh.buf[wid];
        int n0 = 0;
        if (!fallback) {
            // K0: the largest key with at least L slice heads at or above it
            const int L = small_k ? ri.k : kKeepCap;
            uint32_t K0 = 0;
            if (G >= L) {
                uint32_t hk[kMaxGcPerLane];
#pragma unroll
                for (int t = 0; t < kMaxGcPerLane; ++t) {
                    const int s = lane + 32 * t;
                    hk[t] = 0u;
                    if (s < G && __ldcg(&rr[s].nc) >= 1u) hk[t] = cand_key(__ldcg(&rr[s].cand[0]));
                }
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
            const double Te = double(ri.Te);
            const double yA = double(xA) / Te, yB = double(xB) / Te;
            const double y0 = double(m) / Te;
            // completeness of position i: buf[i] lies above every token a slice withheld
            auto complete = [&](int i) { return i < 0 || buf[i] > tau_inc; };
            int np = nk;
            if (ri.do_topp) {
                double Z;
                const double eA = iA < nk ? exp(yA - y0) : 0.0;
                const double eB = iB < nk ? exp(yB - y0) : 0.0;
                double sA = eA, sB = eB;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const double oA = __shfl_up_sync(0xffffffffu, sA, off);
                    const double oB = __shfl_up_sync(0xffffffffu, sB, off);
                    if (lane >= off) {
                        sA += oA;
                        sB += oB;
                    }
                }
                const double totA = __shfl_sync(0xffffffffu, sA, 31);
                sB += totA;
                if (small_k) {
                    Z = __shfl_sync(0xffffffffu, sB, 31);
                } else {
                    // the whole row's mass, from the slices' compensated partial sums
                    double z = 0.0;
                    for (int s = lane; s < G; s += 32) {
                        const float mx = __ldcg(&rr[s].mx);
                        if (!(mx > -INFINITY)) continue;
                        const double zs = double(__ldcg(&rr[s].zs)) - double(__ldcg(&rr[s].zc));
                        z += zs * exp((double(mx) - double(m)) / Te);
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
                    Z = z;
                }
                const double pz = double(ri.p) * Z;
                const bool kA = iA < nk && ((sA - eA) < pz || iA == 0);
                const bool kB = iB < nk && ((sB - eB) < pz);
                np = __popc(__ballot_sync(0xffffffffu, kA)) + __popc(__ballot_sync(0xffffffffu, kB));
                // the list must reach the first dropped token unless top-k closed it
                if (!small_k && np >= lim) fallback = true;
            } else if (!small_k) {
                np = lim;
            }
            int nkept = np;
            if (ri.do_minp) {
                const double th = double(m) + Te * log(double(ri.minp));
                float xthr = float(th);
                if (double(xthr) < th) xthr = nextafterf(xthr, INFINITY);
                const bool mA = iA < np && xA >= xthr;
                const bool mB = iB < np && xB >= xthr;
                nkept = __popc(__ballot_sync(0xffffffffu, mA)) + __popc(__ballot_sync(0xffffffffu, mB));
                nkept = max(nkept, 1);
                if (!small_k && !ri.do_topp && nkept >= lim) fallback = true;
            } else if (!small_k && !ri.do_topp) {
                fallback = true;  // cannot happen for a truncated row; be safe
            }
            if (!fallback) {
                // every kept token must be known exactly, and so must the first dropped
                // one when min-p or top-p (not top-k) closed the set
                if (!complete(nkept - 1)) fallback = true;
                if (small_k && !complete(nk - 1)) fallback = true;
                if (nkept < (small_k ? nk : lim) && !complete(nkept)) fallback = true;
            }
            if (!fallback) {
                const RowParams rp = as_row_params(ri);
                double sa = -INFINITY, sb = -INFINITY;
                if (iA < nkept) sa = gumbel_score_f64(xA, ri.T, noise_word(rp, idxA));
                if (iB < nkept) sb = gumbel_score_f64(xB, ri.T, noise_word(rp, idxB));
                double sc = sa;
                int id = iA < nkept ? idxA : INT_MAX;
                if (iB < nkept && (sb > sc || (sb == sc && idxB < id))) {
                    sc = sb;
                    id = idxB;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const double os = __shfl_xor_sync(0xffffffffu, sc, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, id, off);
                    if (os > sc || (os == sc && oi < id)) {
                        sc = os;
                        id = oi;
                    }
                }
                token = id;
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
    return fallback;
}

template <typename InT>
__global__ void __launch_bounds__(kT, 1) colsplit_kernel(const ColParams P)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    ColShared& sh = *reinterpret_cast<ColShared*>(smem_raw);
    unsigned char* stage = smem_raw + ((sizeof(ColShared) + 127) & ~size_t(127));
    constexpr int ES = int(sizeof(InT));
    const KernelParams& kp = P.k;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int s = blockIdx.x;
    const int N = P.n_rows;
    const int V = int(kp.vocab);
    const int W = P.w;
    const int v0 = s * W;
    const int n = max(0, min(V - v0, W));

    // ---- 1. staging: warp w copies rows w, w + kW, ... of this slice with 16-byte
    // asynchronous copies; each row completes one mbarrier (2 arrivals per lane:
    // one when the lane's copies land, one after its plain edge stores)
    if (tid == 0) sh.n_fallback = 0;
    for (int r = wid; r < N; r += kW) {
        if (lane == 0) mbar_init(&sh.mbar[r], 64);
        __syncwarp();
        const int lrow = kp.logit_row ? kp.logit_row[r] : r;
        const bool lrow_ok = lrow >= 0 && int64_t(lrow) < kp.n_logit_rows;
        int hb = 0, hend = n, tbeg = n;
        if (lrow_ok && n > 0) {
            const unsigned char* g = static_cast<const unsigned char*>(kp.logits) +
                                     (int64_t(lrow) * kp.row_stride + v0) * ES;
            const uintptr_t a = reinterpret_cast<uintptr_t>(g);
            hb = int(a & 15u);
            const uintptr_t A0 = (a + 15u) & ~uintptr_t(15);
            const uintptr_t A1 = (a + uintptr_t(n) * ES) & ~uintptr_t(15);
            unsigned char* dst = stage + size_t(r) * P.row_bytes + hb;  // element i at dst + i * ES
            if (A1 > A0) {
                hend = int((A0 - a) / ES);
                tbeg = int((A1 - a) / ES);
                const int nv = int((A1 - A0) / 16);
                unsigned char* d16 = dst + (A0 - a);
                for (int q = lane; q < nv; q += 32)
                    cp_async16(d16 + 16 * q, reinterpret_cast<const void*>(A0 + 16 * size_t(q)));
            }
            const InT* ge = reinterpret_cast<const InT*>(g);
            InT* de = reinterpret_cast<InT*>(dst);
            for (int i = lane; i < hend; i += 32) de[i] = ge[i];
            for (int i = tbeg + lane; i < n; i += 32) de[i] = ge[i];
        }
        cp_async_arrive_noinc(&sh.mbar[r]);
        mbar_arrive_release(&sh.mbar[r]);
        if (lane == 0) {
            sh.info[r].lrow = lrow;
            sh.info[r].status = lrow_ok ? kRowOk : kRowBadParam;
            sh.info[r].hb = hb;
            sh.info[r].head_end = hend;
            sh.info[r].tail_begin = tbeg;
        }
    }
    __syncthreads();
    // ---- 2. row parameters (while the copies are in flight)
    for (int r = tid; r < N; r += kT) {
        RowInfo ri = sh.info[r];
        const int lrow = ri.lrow;
        const bool lrow_ok = ri.status == kRowOk;
        const int hb = ri.hb, hend = ri.head_end, tbeg = ri.tail_begin;
        load_row_info(P, r, lrow, lrow_ok, ri);
        ri.hb = hb;
        ri.head_end = hend;
        ri.tail_begin = tbeg;
        sh.info[r] = ri;
    }
    __syncthreads();

    // ---- 3. cost-ordered, snake-assigned rows per warp
    __shared__ int16_t wl[kW][kMaxRows / kW + 1];
    __shared__ int16_t wcnt[kW];
    __shared__ int16_t wsplit[kW];
    __shared__ int wcnt_i[kW];
    if (tid < kW) wcnt_i[tid] = 0;
    __syncthreads();
    if (wid == 0) {
        // balance by cost: plain, truncated, greedy, error -- snake over the warps
        const uint8_t cost_order[4] = {kClsPlain, kClsCand, kClsGreedy, kClsErr};
        int j = 0;
        for (int c = 0; c < 4; ++c) {
            for (int r0 = 0; r0 < N; r0 += 32) {
                const int r = r0 + lane;
                const bool pred = r < N && sh.info[r].cls == cost_order[c];
                const unsigned bal = __ballot_sync(0xffffffffu, pred);
                if (pred) {
                    const int pos = j + __popc(bal & ((1u << lane) - 1u));
                    const int lap = pos / kW, q = pos % kW;
                    sh.warp_of[r] = int16_t((lap & 1) ? (kW - 1 - q) : q);
                }
                j += __popc(bal);
            }
        }
        __syncwarp();
        // within a warp: truncated rows first (their finishing overlaps the rest),
        // then errors, plain, greedy
        const uint8_t run_order[4] = {kClsCand, kClsErr, kClsPlain, kClsGreedy};
        for (int c = 0; c < 4; ++c) {
            for (int r0 = 0; r0 < N; r0 += 32) {
                const int r = r0 + lane;
                if (r < N && sh.info[r].cls == run_order[c]) {
                    const int w = sh.warp_of[r];
                    const int pos = atomicAdd(&wcnt_i[w], 1);
                    wl[w][pos] = int16_t(r);
                }
            }
            __syncwarp();
            if (c == 0 && lane < kW) wsplit[lane] = int16_t(wcnt_i[lane]);
            __syncwarp();
        }
        if (lane < kW) wcnt[lane] = int16_t(wcnt_i[lane]);
    }
    __syncthreads();

    // ---- 4. phase A and finishing, per warp
    const int nmine = wcnt[wid];
    const int split = wsplit[wid];
    int batch_begin = 0;
    for (int t = 0; t < nmine; ++t) {
        const int r = wl[wid][t];
        const RowInfo& ri = sh.info[r];
        SliceView<InT> sv;
        sv.st = stage + size_t(r) * P.row_bytes;
        sv.hoff = ri.hb / ES;
        sv.n = (ri.status == kRowOk) ? n : 0;
        sv.v0 = v0;
        slice_summary<InT>(P, sh, r, sv, P.rec + int64_t(r) * P.gc + s);
        const bool end_batch = (t == split - 1) || (t == nmine - 1);
        if (!end_batch) continue;
        // publish this batch, then count arrivals
        __threadfence();
        __syncwarp();
        const int nb = t + 1 - batch_begin;
        unsigned last_mask = 0;
        for (int b0 = 0; b0 < nb; b0 += 32) {
            bool last = false;
            if (b0 + lane < nb) {
                const int rr = wl[wid][batch_begin + b0 + lane];
                last = atomicAdd(&P.counters[rr], 1u) == uint32_t(P.gc - 1);
            }
            const unsigned bm = __ballot_sync(0xffffffffu, last);
            for (unsigned m2 = bm; m2; m2 &= m2 - 1) {
                const int bb = b0 + __ffs(m2) - 1;
                const int rr = wl[wid][batch_begin + bb];
                float mrow;
                int arow;
                const bool fb = finish_row<InT>(P, sh, rr, mrow, arow);
                if (fb && lane == 0) {
                    const int q = atomicAdd(&sh.n_fallback, 1);
                    sh.fallback_rows[q] = rr;
                    sh.fb_m[q] = mrow;
                    sh.fb_amax[q] = arow;
                }
                __syncwarp();
            }
            (void)last_mask;
        }
        batch_begin = t + 1;
    }
    __syncthreads();

    // ---- 5. rows the candidates could not settle: exact path, whole CTA
    const int nf = sh.n_fallback;
    if (tid == 0 && nf > 0 && P.stats) atomicAdd(&P.stats[0], (unsigned long long)nf);
    for (int q = 0; q < nf; ++q)
        cta_exact_row<InT>(sh, P, sh.fallback_rows[q], sh.fb_m[q], sh.fb_amax[q]);
}

}  // namespace col
}  // namespace dst
