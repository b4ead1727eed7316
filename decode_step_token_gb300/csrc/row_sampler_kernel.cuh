// row_sampler_kernel.cuh -- the kernel body (see row_sampler.cuh for the design).
#pragma once

#include "row_sampler.cuh"

namespace dst {

__device__ __forceinline__ int align16i(int x) { return (x + 15) & ~15; }

// Element i of the slice as a penalised fp32 logit.
template <typename InT, bool kPen>
__device__ __forceinline__ float slice_x(const Slice& sl, const RowParams& rp, int i)
{
    const unsigned char* p = sl.stage + (sl.hoff + i) * int(sizeof(InT));
    float x;
    if (sizeof(InT) == 4)
        x = *reinterpret_cast<const float*>(p);
    else
        x = __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(p)) << 16);
    if (kPen && rp.has_hist) {
        const uint32_t c = sl.cnt[i];
        if (c) x = penalize(x, c, rp);
    }
    return x;
}

__device__ __forceinline__ void bitonic_sort_desc(unsigned long long* a, int n)
{
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = threadIdx.x; t < (n >> 1); t += kThreads) {
                const int lo = 2 * stride * (t / stride) + (t % stride);
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long x = a[lo], y = a[hi];
                if ((x < y) == desc) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

// Write the fields a radix level (or the tie search) changed into every CTA.
__device__ __forceinline__ void bcast_radix_state(Shared& sh, uint32_t C)
{
    const int t = threadIdx.x;
    if (t < int(C)) {
        const uint32_t rank = uint32_t(t);
        dsmem_st_u32(dsmem_map(smem_addr(&sh.bc.prefix), rank), sh.bc.prefix);
        dsmem_st_u32(dsmem_map(smem_addr(&sh.bc.pbits), rank), sh.bc.pbits);
        dsmem_st_u64(dsmem_map(smem_addr(&sh.bc.w_above), rank), sh.bc.w_above);
        dsmem_st_u64(dsmem_map(smem_addr(&sh.bc.target), rank), sh.bc.target);
        dsmem_st_u32(dsmem_map(smem_addr(&sh.bc.tie_cta), rank), uint32_t(sh.bc.tie_cta));
        dsmem_st_u32(dsmem_map(smem_addr(&sh.bc.tie_j), rank), uint32_t(sh.bc.tie_j));
    }
}

// Cluster-wide selection of the kept prefix in (value desc, index asc) order.
// Weights are 1 per token (count mode, target = k) or the fixed-point softmax
// mass (mass mode, target = ceil(p * total mass of the domain)). The kept prefix
// ends at the first token whose inclusive weight reaches the target. Tokens
// outside the domain prefix (dkey, didx) weigh nothing. Returns the last kept
// token as (key, index). Every CTA of the cluster calls this.
template <typename InT, bool kPen>
__device__ void radix_select(Shared& sh, const Slice& sl, const RowParams& rp, uint32_t rank,
                             uint32_t C, bool mass_mode, bool dom, uint32_t dkey, int didx,
                             float m, unsigned long long count_target, uint32_t& out_key,
                             int& out_idx)
{
    const int tid = threadIdx.x;
    if (tid == 0) {
        sh.bc.prefix = 0;
        sh.bc.pbits = 0;
        sh.bc.w_above = 0;
        sh.bc.target = count_target;
        sh.bc.tie_cta = -1;
        sh.bc.tie_j = 0;
    }
    __syncthreads();
    for (int level = 0; level < 4; ++level) {
        for (int i = tid; i < 256; i += kThreads) {
            sh.hcnt[i] = 0;
            sh.hmass[i] = 0;
        }
        __syncthreads();
        const uint32_t prefix = sh.bc.prefix, pbits = sh.bc.pbits;
        const int shift = 24 - 8 * level;
        for_each<InT, kPen>(sl, rp, [&](int v, float x) {
            const uint32_t key = f2key(x);
            if (dom && !in_prefix(key, v, dkey, didx)) return;
            if (pbits && (key >> (32 - pbits)) != prefix) return;
            const uint32_t d = (key >> shift) & 255u;
            atomicAdd(&sh.hcnt[d], 1u);
            if (mass_mode) atomicAdd(&sh.hmass[d], mass_q(x, m, rp.invT));
        });
        __syncthreads();
        cluster_sync();
        if (rank == 0) {
            const int d = tid;  // one thread per digit
            unsigned long long tc = 0, tm = 0;
            for (uint32_t c = 0; c < C; ++c) {
                tc += dsmem_ld_u32(dsmem_map(smem_addr(&sh.hcnt[d]), c));
                if (mass_mode) tm += dsmem_ld_u64(dsmem_map(smem_addr(&sh.hmass[d]), c));
            }
            const unsigned long long wgt = mass_mode ? tm : tc;
            const unsigned long long incl = block_suffix_scan(wgt, sh);
            if (tid == 0) sh.red_z[0] = incl;  // total weight
            __syncthreads();
            unsigned long long target = sh.bc.target;
            if (mass_mode && level == 0) {
                const double z = double(sh.red_z[0]);
                target = (unsigned long long)ceil(double(rp.p) * z);
                if (target < 1) target = 1;
            }
            const unsigned long long above = incl - wgt;
            const unsigned long long wa = sh.bc.w_above;
            __syncthreads();
            if (tid == 0) sh.bc.target = target;
            if (wa + incl >= target && wa + above < target) {
                const uint32_t np = (prefix << 8) | uint32_t(d);
                const unsigned long long nwa = wa + above;
                sh.bc.prefix = np;
                sh.bc.pbits = pbits + 8;
                sh.bc.w_above = nwa;
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
                    sh.bc.tie_cta = cstar;
                    sh.bc.tie_j = int(jloc);
                }
            }
            __syncthreads();
            bcast_radix_state(sh, C);
        }
        cluster_sync();
    }

    // the tie_j-th token (in index order) carrying the boundary key
    const uint32_t K = sh.bc.prefix;
    if (int(rank) == sh.bc.tie_cta) {
        constexpr int EPV = ElemTraits<InT>::kPerVec;
        const int nvec = (sl.hoff + sl.n + EPV - 1) / EPV;
        const int need = sh.bc.tie_j;
        int base = 0;
        for (int j0 = 0; j0 < nvec; j0 += kThreads) {
            const int j = j0 + tid;
            int cntv = 0;
            if (j < nvec) {
                for (int e = 0; e < EPV; ++e) {
                    const int i = j * EPV + e - sl.hoff;
                    if (i < 0 || i >= sl.n) continue;
                    const float x = slice_x<InT, kPen>(sl, rp, i);
                    const uint32_t key = f2key(x);
                    if (key == K && (!dom || in_prefix(key, sl.v0 + i, dkey, didx))) ++cntv;
                }
            }
            int total = 0;
            const int excl = block_excl_scan(cntv, total, sh);
            if (cntv > 0 && need > base + excl && need <= base + excl + cntv) {
                int left = need - base - excl;
                for (int e = 0; e < EPV; ++e) {
                    const int i = j * EPV + e - sl.hoff;
                    if (i < 0 || i >= sl.n) continue;
                    const float x = slice_x<InT, kPen>(sl, rp, i);
                    const uint32_t key = f2key(x);
                    if (key == K && (!dom || in_prefix(key, sl.v0 + i, dkey, didx))) {
                        if (--left == 0) {
                            for (uint32_t c = 0; c < C; ++c)
                                dsmem_st_u32(dsmem_map(smem_addr(&sh.bc.bidx), c), uint32_t(sl.v0 + i));
                            break;
                        }
                    }
                }
            }
            base += total;
            if (base >= need) break;
        }
    }
    cluster_sync();
    out_key = K;
    out_idx = sh.bc.bidx;
}

template <typename InT, bool kPen>
__global__ void __launch_bounds__(kThreads, 1) row_sampler_kernel(const KernelParams P)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
    constexpr int ES = int(sizeof(InT));
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const uint32_t C = cluster_nctarank();
    const int r = int(cluster_id_x());
    const int V = int(P.vocab);
    const int L = P.slice_len;
    const int v0 = int(rank) * L;
    const int n = max(0, min(V - v0, L));

    unsigned char* after = smem_raw + align16i(int(sizeof(Shared)));
    uint16_t* cnt = kPen ? reinterpret_cast<uint16_t*>(after) : nullptr;
    unsigned char* stage = after + (kPen ? align16i(L * 2 + 4) : 0);

    __shared__ int s_nchunks, s_hb, s_head_end, s_tail_begin;

    // ---- set-up: bulk copies first, then the row's parameters
    if (tid == 0) {
        for (int c = 0; c < kChunks; ++c) mbar_init(&sh.mbar[c], 1);
        fence_mbar_init();
        const int lrow = P.logit_row ? P.logit_row[r] : r;
        const bool lrow_ok = lrow >= 0 && int64_t(lrow) < P.n_logit_rows;
        int nch = 0, hb = 0, head_end = n, tail_begin = n;
        if (lrow_ok && n > 0) {
            const unsigned char* g = static_cast<const unsigned char*>(P.logits) +
                                     (int64_t(lrow) * P.row_stride + v0) * ES;
            const uintptr_t a = reinterpret_cast<uintptr_t>(g);
            hb = int(a & 15u);
            const uintptr_t A0 = (a + 15u) & ~uintptr_t(15);
            const uintptr_t A1 = (a + uintptr_t(n) * ES) & ~uintptr_t(15);
            if (A1 > A0) {
                head_end = int((A0 - a) / ES);
                tail_begin = int((A1 - a) / ES);
                const uint32_t bytes = uint32_t(A1 - A0);
                const uint32_t per = ((bytes / kChunks) + 15u) & ~15u;
                uint32_t done = 0;
                while (done < bytes && nch < kChunks) {
                    const uint32_t b = min(per ? per : bytes, bytes - done);
                    mbar_arrive_expect_tx(&sh.mbar[nch], b);
                    bulk_copy_g2s(stage + (A0 - (a - hb)) + done, reinterpret_cast<const void*>(A0 + done),
                                  b, &sh.mbar[nch]);
                    done += b;
                    ++nch;
                }
            }
        }
        s_nchunks = nch;
        s_hb = hb;
        s_head_end = head_end;
        s_tail_begin = tail_begin;
        read_row_params(P, r, sh.rp);
        if (!lrow_ok) sh.rp.status = kRowBadParam;
        sh.part.flags = 0;
    }
    __syncthreads();
    const RowParams rp = sh.rp;
    Slice sl;
    sl.stage = stage;
    sl.cnt = cnt;
    sl.n = n;
    sl.hoff = s_hb / ES;
    sl.v0 = v0;

    // head / tail elements outside the 16-byte-aligned interior: plain loads
    if (rp.status == kRowOk && n > 0) {
        const unsigned char* g = static_cast<const unsigned char*>(P.logits) +
                                 (int64_t(rp.lrow) * P.row_stride + v0) * ES;
        const int hend = s_head_end, tbeg = s_tail_begin;
        auto copy1 = [&](int i) {
            if (ES == 4)
                reinterpret_cast<float*>(stage + s_hb)[i] = reinterpret_cast<const float*>(g)[i];
            else
                reinterpret_cast<uint16_t*>(stage + s_hb)[i] = reinterpret_cast<const uint16_t*>(g)[i];
        };
        for (int i = tid; i < hend; i += kThreads) copy1(i);
        for (int i = tbeg + tid; i < n; i += kThreads) copy1(i);
    }

    // history counts of this slice (penalties)
    bool bad_hist = false;
    if (kPen && rp.has_hist && rp.status == kRowOk) {
        uint4* c4 = reinterpret_cast<uint4*>(cnt);
        const int nw4 = (L * 2 + 15) / 16;
        for (int i = tid; i < nw4; i += kThreads) c4[i] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        const int len = rp.hhi - rp.hlo;
        if (len < 0 || len > 65535) {
            bad_hist = true;
        } else {
            uint32_t* c32 = reinterpret_cast<uint32_t*>(cnt);
            for (int j = rp.hlo + tid; j < rp.hhi; j += kThreads) {
                const int id = P.hist_ids[j];
                if (id < 0 || id >= V) {
                    bad_hist = true;
                } else if (id >= v0 && id < v0 + n) {
                    const int i = id - v0;
                    atomicAdd(&c32[i >> 1], 1u << (16 * (i & 1)));
                }
            }
        }
    }
    bad_hist = __syncthreads_or(bad_hist);

    // wait for the bulk copies (bounded)
    bool timeout = false;
    for (int c = 0; c < s_nchunks; ++c)
        if (!mbar_wait_bounded(&sh.mbar[c], 0, kMaxPolls)) timeout = true;
    timeout = __syncthreads_or(timeout);

    // ---- P1: max / argmax / non-finite; the Gumbel pick of plain rows
    float mx = -INFINITY;
    int am = INT_MAX;
    bool nonfin = false, anyfin = false;
    GumbelAcc g;
    gumbel_init(g);
    const bool ok0 = rp.status == kRowOk && !bad_hist && !timeout;
    const bool g1 = ok0 && rp.plain_single;
    if (ok0) {
        for_each<InT, kPen>(sl, rp, [&](int v, float x) {
            if (x != x || x == INFINITY) nonfin = true;
            else if (x > -INFINITY) anyfin = true;
            if (x > mx) {
                mx = x;
                am = v;
            }
            if (g1) gumbel_visit(g, rp, v, x);
        });
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, off);
        const int oi = __shfl_xor_sync(0xffffffffu, am, off);
        maxidx_merge(mx, am, om, oi);
    }
    const bool wnf = __any_sync(0xffffffffu, nonfin), waf = __any_sync(0xffffffffu, anyfin);
    if (g1) top2_warp_reduce(g.t);
    if (lane == 0) {
        sh.red_f[wid] = mx;
        sh.red_i[wid] = am;
        sh.red_u[wid] = (wnf ? kFlagNonFinite : 0u) | (waf ? kFlagAnyFinite : 0u);
        sh.red_g[wid] = g.t;
    }
    __syncthreads();
    if (tid == 0) {
        float m = -INFINITY;
        int a = INT_MAX;
        uint32_t fl = (bad_hist ? kFlagBadHistory : 0u) | (timeout ? kFlagTimeout : 0u);
        GTop2 t;
        t.a = grec_empty();
        t.b = grec_empty();
        for (int w = 0; w < kWarps; ++w) {
            maxidx_merge(m, a, sh.red_f[w], sh.red_i[w]);
            fl |= sh.red_u[w];
            sh.part.wmax[w] = sh.red_f[w];
            if (g1) {
                top2_insert(t, sh.red_g[w].a);
                top2_insert(t, sh.red_g[w].b);
            }
        }
        sh.part.mx = m;
        sh.part.amax = a;
        sh.part.flags = fl;
        sh.part.g0 = t.a;
        sh.part.g1 = t.b;
    }
    __syncthreads();
    cluster_sync();

    // ---- R1 (leader): status, max, early picks, selection plan
    if (rank == 0 && wid == 0) {
        const bool have = lane < int(C);
        Partial q;
        if (have) dsmem_read(q, sh.part, uint32_t(lane));
        float m = have ? q.mx : -INFINITY;
        int a = have ? q.amax : INT_MAX;
        uint32_t fl = have ? q.flags : 0u;
        GTop2 t;
        t.a = have ? q.g0 : grec_empty();
        t.b = have ? q.g1 : grec_empty();
        if (have)
            for (int w = 0; w < kWarps; ++w) sh.wm_all[lane * kWarps + w] = q.wmax[w];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, off);
            const int oi = __shfl_xor_sync(0xffffffffu, a, off);
            maxidx_merge(m, a, om, oi);
            fl |= __shfl_xor_sync(0xffffffffu, fl, off);
        }
        if (rp.plain_single) top2_warp_reduce(t);
        __syncwarp();

        Bcast b;
        b.status = rp.status;
        if (b.status == kRowOk) {
            if (fl & kFlagBadHistory) b.status = kRowBadHistory;
            else if (fl & kFlagTimeout) b.status = kRowTimeout;
            else if (fl & kFlagNonFinite) b.status = kRowNonFinite;
            else if (!(fl & kFlagAnyFinite)) b.status = kRowAllNegInf;
        }
        b.done = 0;
        b.token = -1;
        b.sel = kSelNone;
        b.m = m;
        b.xthr = -INFINITY;
        b.tau = -INFINITY;
        b.lnz = 0.0f;
        b.bkey = 0;
        b.bidx = 0;
        b.has_bound = 0;
        b.prefix = 0;
        b.pbits = 0;
        b.tie_cta = -1;
        b.tie_j = 0;
        b.amax = a;
        b.w_above = 0;
        b.target = 0;
        if (b.status != kRowOk) {
            b.done = 1;
        } else if (rp.greedy && !rp.want_out) {
            b.token = a;
            b.done = 1;
        } else if (rp.plain_single) {
            b.token = settle_top2(t, rp.T);
            b.done = 1;
        } else {
            if (rp.do_minp) {
                const double th = double(m) + double(rp.Te) * log(double(rp.minp));
                float f = float(th);
                if (double(f) < th) f = nextafterf(f, INFINITY);
                b.xthr = f;
            }
            const int nw = int(C) * kWarps;
            if (rp.do_topk && rp.k <= nw) {
                // k-th largest warp maximum: at least k tokens reach it
                float tau = -INFINITY;
                bool found = false;
                for (int i = lane; i < nw; i += 32) {
                    const float wi = sh.wm_all[i];
                    int rk = 0;
                    for (int j = 0; j < nw; ++j) {
                        const float wj = sh.wm_all[j];
                        rk += (wj > wi) || (wj == wi && j < i);
                    }
                    if (rk == rp.k - 1) {
                        tau = wi;
                        found = true;
                    }
                }
                const unsigned bal = __ballot_sync(0xffffffffu, found);
                tau = __shfl_sync(0xffffffffu, tau, __ffs(bal) - 1);
                b.tau = rp.do_topp ? tau : fmaxf(tau, b.xthr);
                b.sel = kSelCand;
            } else if (rp.do_topk || rp.do_topp) {
                b.sel = kSelRadix;
            }
        }
        if (have) dsmem_write(b, sh.bc, uint32_t(lane));
    }
    cluster_sync();

    Bcast bc = sh.bc;
    auto finish = [&](const Bcast& fb) {
        if (rank == 0 && tid == 0) {
            P.out_tokens[r] = fb.token;
            if (P.out_status) P.out_status[r] = fb.status;
        }
    };
    auto fill_nan = [&]() {
        for (int i = tid; i < n; i += kThreads) {
            const int64_t o = int64_t(r) * V + v0 + i;
            if (P.out_probs) P.out_probs[o] = __int_as_float(0x7fc00000);
            if (P.out_logprobs) P.out_logprobs[o] = __int_as_float(0x7fc00000);
        }
    };
    if (bc.done) {
        finish(bc);
        if (bc.status != kRowOk && rp.want_out) fill_nan();
        return;
    }

    const float m = bc.m;
    const float xthr = bc.xthr;

    // ---- candidate path: tokens >= tau hold the whole kept set
    if (bc.sel == kSelCand) {
        if (tid == 0) sh.ncand = 0;
        __syncthreads();
        const float tau = bc.tau;
        for_each<InT, kPen>(sl, rp, [&](int v, float x) {
            if (x >= tau) {
                const uint32_t pos = atomicAdd(&sh.ncand, 1u);
                if (pos < uint32_t(kCandPerCta)) sh.cand[pos] = cand_word(f2key(x), v);
            }
        });
        __syncthreads();
        if (tid == 0) sh.part.ncand = sh.ncand;
        __syncthreads();
        cluster_sync();
        if (rank == 0) {
            uint32_t counts[kMaxCluster];
            uint32_t total = 0;
            bool overflow = false;
            for (uint32_t c = 0; c < C; ++c) {
                counts[c] = dsmem_ld_u32(dsmem_map(smem_addr(&sh.part.ncand), c));
                overflow |= counts[c] > uint32_t(kCandPerCta);
                total += counts[c];
            }
            overflow |= total > uint32_t(kCandTotal);
            Bcast b = bc;
            if (!overflow) {
                uint32_t off = 0;
                for (uint32_t c = 0; c < C; ++c) {
                    for (uint32_t i = tid; i < counts[c]; i += kThreads)
                        sh.sortbuf[off + i] = dsmem_ld_u64(dsmem_map(smem_addr(&sh.cand[i]), c));
                    off += counts[c];
                }
                int np2 = 1;
                while (np2 < int(total)) np2 <<= 1;
                for (int i = int(total) + tid; i < np2; i += kThreads) sh.sortbuf[i] = 0ull;
                __syncthreads();
                bitonic_sort_desc(sh.sortbuf, np2);
                if (wid == 0) {
                    const int ns = int(total);
                    const int nk = min(rp.k, ns);  // k <= 64 on this path
                    const int iA = lane, iB = lane + 32;
                    const unsigned long long cA = iA < nk ? sh.sortbuf[iA] : 0ull;
                    const unsigned long long cB = iB < nk ? sh.sortbuf[iB] : 0ull;
                    const float xA = key2f(cand_key(cA)), xB = key2f(cand_key(cB));
                    const int idxA = cand_idx(cA), idxB = cand_idx(cB);
                    const double Te = double(rp.Te);
                    const double yA = double(xA) / Te, yB = double(xB) / Te;
                    const double y0 = __shfl_sync(0xffffffffu, yA, 0);
                    int np = nk;
                    if (rp.do_topp) {
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
                        const double Z = __shfl_sync(0xffffffffu, sB, 31);
                        const double pz = double(rp.p) * Z;
                        const bool kA = iA < nk && ((sA - eA) < pz || iA == 0);
                        const bool kB = iB < nk && ((sB - eB) < pz);
                        np = __popc(__ballot_sync(0xffffffffu, kA)) + __popc(__ballot_sync(0xffffffffu, kB));
                    }
                    int nkept = np;
                    if (rp.do_minp) {
                        const bool mA = iA < np && xA >= xthr;
                        const bool mB = iB < np && xB >= xthr;
                        nkept = __popc(__ballot_sync(0xffffffffu, mA)) + __popc(__ballot_sync(0xffffffffu, mB));
                        nkept = max(nkept, 1);
                    }
                    int token = bc.amax;
                    if (!rp.greedy) {
                        double sa = -INFINITY, sb = -INFINITY;
                        if (iA < nkept) sa = gumbel_score_f64(xA, rp.T, noise_word(rp, idxA));
                        if (iB < nkept) sb = gumbel_score_f64(xB, rp.T, noise_word(rp, idxB));
                        double s = sa;
                        int id = iA < nkept ? idxA : INT_MAX;
                        if (iB < nkept && (sb > s || (sb == s && idxB < id))) {
                            s = sb;
                            id = idxB;
                        }
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) {
                            const double os = __shfl_xor_sync(0xffffffffu, s, off);
                            const int oi = __shfl_xor_sync(0xffffffffu, id, off);
                            if (os > s || (os == s && oi < id)) {
                                s = os;
                                id = oi;
                            }
                        }
                        token = id;
                    }
                    double zk = (iA < nkept ? exp(yA - y0) : 0.0) + (iB < nkept ? exp(yB - y0) : 0.0);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) zk += __shfl_xor_sync(0xffffffffu, zk, off);
                    const unsigned long long cl = sh.sortbuf[nkept - 1];
                    b.token = token;
                    b.lnz = float(log(zk));
                    b.bkey = cand_key(cl);
                    b.bidx = cand_idx(cl);
                    b.has_bound = 1;
                    b.sel = kSelCand;
                    b.done = rp.want_out ? 0 : 1;
                    if (lane == 0) sh.bc = b;
                }
            } else {
                if (tid == 0) {
                    b.sel = kSelRadix;
                    sh.bc = b;
                }
            }
            __syncthreads();
            if (tid < int(C)) dsmem_write(sh.bc, sh.bc, uint32_t(tid));
        }
        cluster_sync();
        bc = sh.bc;
        if (bc.done) {
            finish(bc);
            return;
        }
    }

    // ---- radix path
    if (bc.sel == kSelRadix) {
        uint32_t bk = 0;
        int bi = 0;
        bool dom = false;
        if (rp.do_topk) {
            radix_select<InT, kPen>(sh, sl, rp, rank, C, false, false, 0u, 0, m,
                                    (unsigned long long)rp.k, bk, bi);
            dom = true;
        }
        if (rp.do_topp) {
            radix_select<InT, kPen>(sh, sl, rp, rank, C, true, dom, bk, bi, m, 0ull, bk, bi);
        }
        bc.bkey = bk;
        bc.bidx = bi;
        bc.has_bound = 1;
    }

    // ---- P3: Gumbel-max over the kept set and its mass
    if (bc.sel != kSelCand) {
        GumbelAcc g3;
        gumbel_init(g3);
        unsigned long long zq = 0;
        const bool hb = bc.has_bound != 0;
        const uint32_t bkey = bc.bkey;
        const int bidx = bc.bidx;
        for_each<InT, kPen>(sl, rp, [&](int v, float x) {
            if (!(x > -INFINITY)) return;
            if (hb && !in_prefix(f2key(x), v, bkey, bidx)) return;
            if (rp.do_minp && !(x >= xthr)) return;
            if (!rp.greedy) gumbel_visit(g3, rp, v, x);
            if (rp.want_out) zq += mass_q(x, m, rp.invT);
        });
        if (!rp.greedy) top2_warp_reduce(g3.t);
        zq = warp_sum_u64(zq);
        if (lane == 0) {
            sh.red_g[wid] = g3.t;
            sh.red_z[wid] = zq;
        }
        __syncthreads();
        if (tid == 0) {
            GTop2 t;
            t.a = grec_empty();
            t.b = grec_empty();
            unsigned long long z = 0;
            for (int w = 0; w < kWarps; ++w) {
                top2_insert(t, sh.red_g[w].a);
                top2_insert(t, sh.red_g[w].b);
                z += sh.red_z[w];
            }
            sh.part.g0 = t.a;
            sh.part.g1 = t.b;
            sh.part.zq = z;
        }
        __syncthreads();
        cluster_sync();
        if (rank == 0 && wid == 0) {
            const bool have = lane < int(C);
            GTop2 t;
            t.a = grec_empty();
            t.b = grec_empty();
            unsigned long long z = 0;
            if (have) {
                Partial q;
                dsmem_read(q, sh.part, uint32_t(lane));
                t.a = q.g0;
                t.b = q.g1;
                z = q.zq;
            }
            top2_warp_reduce(t);
            z = warp_sum_u64(z);
            Bcast b = bc;
            b.token = rp.greedy ? bc.amax : settle_top2(t, rp.T);
            b.lnz = float(log(double(z)) - 40.0 * 0.69314718055994530942);
            if (have) dsmem_write(b, sh.bc, uint32_t(lane));
        }
        cluster_sync();
        bc = sh.bc;
    }

    finish(bc);

    // ---- P4: fp32 probs / logprobs of the kept set
    if (rp.want_out) {
        const bool hb = bc.has_bound != 0;
        const float lnz = bc.lnz;
        const float Te = rp.Te;
        for (int i = tid; i < n; i += kThreads) {
            const int v = v0 + i;
            const float x = slice_x<InT, kPen>(sl, rp, i);
            bool kept = x > -INFINITY;
            if (kept && hb) kept = in_prefix(f2key(x), v, bc.bkey, bc.bidx);
            if (kept && rp.do_minp) kept = x >= xthr;
            float lp = -INFINITY, pr = 0.0f;
            if (kept) {
                lp = __fdiv_rn(x - m, Te) - lnz;
                pr = expf(lp);
            }
            const int64_t o = int64_t(r) * V + v;
            if (P.out_probs) P.out_probs[o] = pr;
            if (P.out_logprobs) P.out_logprobs[o] = lp;
        }
    }
}

}  // namespace dst
