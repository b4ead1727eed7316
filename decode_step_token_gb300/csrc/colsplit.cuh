// colsplit.cuh -- the unit-split sampler kernel for small batches (sm_103a).
//
// Each row is cut into G equal vocabulary units, and the N x G units are spread
// over every warp of a cooperative grid (one CTA of 16 warps per SM), one unit
// per warp when the batch allows. The kernel runs in two phases; a row's
// phase 2 starts once all of that row's units are done (no grid-wide barrier):
//
//   phase 1  a warp copies its unit into its own shared-memory slot (16-byte
//            cp.async copies in four groups; work starts on the first while the
//            rest land) and writes a summary record of the unit:
//              greedy rows     the unit's maximum and its lowest index
//              plain rows      the unit's best two Gumbel scores (fp32)
//              truncated rows  tau, the C-th largest of 128 group maxima
//                              (C = k when k <= 64, else 64), and every token
//                              of the unit at or above it (unsorted; at least
//                              C of them, so the unit's top C are among them)
//   phase 2  rows are dealt round-robin to the CTAs. A greedy or plain row is
//            finished by one warp from its G records (the best two Gumbel
//            scores settled in double). A truncated row is finished by the whole
//            CTA: every listed token at or above the largest tau of the row is
//            gathered -- exactly the row's tokens above that value, which hold
//            its top C -- ranked, then top-k / top-p / min-p are cut in double
//            and the Gumbel-max pick is taken over the kept tokens.
//
// A truncated row whose kept set reaches below what the lists cover is sampled
// exactly by its phase-2 CTA, streaming the row from global memory (radix
// select by count or fixed-point softmax mass, then a Gumbel pass). A row's
// finishing CTA waits only for that row: every unit adds one to the row's
// counter once its record is written (release), and the finisher polls it
// (acquire) until all G units are in, then sets it back to zero. The cooperative
// launch keeps every CTA resident, so each wait ends; it gives up after a
// bounded number of polls and marks the row SAMPLER_ROW_TIMEOUT.
#pragma once

#include "row_sampler.cuh"

namespace dst {
namespace col {

constexpr int kT = 512;
constexpr int kW = kT / 32;
constexpr int kSlotBytes = 9216;   // staged logits per warp: 4608 bf16 or 2304 fp32
constexpr int kSeg = 16;           // candidate words a lane may hold in phase 1
constexpr int kBufCap = 32 * kSeg;
constexpr int kUnitCands = 128;    // tokens a unit may gather at or above its tau
constexpr int kCandCap = 64;       // top list of a row without a small top-k
constexpr int kKeepCap = 64;       // kept tokens a finishing warp resolves
constexpr int kSelCap = 512;       // tokens a phase-2 CTA gathers for one row
constexpr int kStages = 4;         // copy groups per unit
constexpr int kMaxRows = 256;
constexpr uint32_t kOverflow = 0xFFFFFFFFu;
constexpr int kUnitMinElems = 2048;  // smallest unit, unless a row is narrower
constexpr int kMaxUnits = 128;       // units per row: 262144 / kUnitMinElems
constexpr int kLPL = kMaxUnits / 32; // a finishing warp's records per lane

enum : uint8_t { kClsErr = 0, kClsGreedy = 1, kClsPlain = 2, kClsCand = 3 };

struct alignas(16) ColRec {  // one (row, unit) summary
    float mx;      // unit maximum (NaN ignored)
    int32_t amax;  // its lowest index
    uint32_t flags;
    uint32_t nc;   // candidates listed, kOverflow if they did not fit
    GRec g0, g1;   // plain rows: the unit's best two Gumbel scores
    float zs;      // top-p rows without top-k: sum of exp((x - mx) / T), compensated
    float zc;      // its compensation term
    uint32_t tau;  // truncated rows: order key of the C-th largest group maximum
    uint32_t pad;
    unsigned long long cand[kCandCap];  // truncated rows: the unit's top list, descending
};

struct RowSync {                // zero-initialised once; every launch leaves it zero
    uint32_t done[kMaxRows];    // units of each row whose record is written
    uint32_t poison;            // set when a wait gave up: later waits fail at once
    uint32_t pad[3];
};

struct ColParams {
    KernelParams k;
    int32_t n_rows;
    int32_t gc;       // units per row
    int32_t w;        // elements per unit (a multiple of 16 bytes)
    int32_t n_units;  // n_rows * gc
    ColRec* rec;      // [n_rows][gc]
    RowSync* sync;
    unsigned long long* stats;  // [0] rows finished by the exact path (diagnostic)
};

struct alignas(16) RowInfo {
    float T, Te, invT, p, minp;
    int32_t k;
    uint32_t stream, key_lo, key_hi, off_lo, off_hi;
    int32_t lrow;
    int32_t status;
    uint8_t cls, do_topk, do_topp, do_minp;
    uint8_t need_z, small_k, greedy, pad;
};

struct alignas(16) ColShared {
    int32_t fallback_rows[kMaxRows];  // rows for the exact path, with their max / argmax
    float fb_m[kMaxRows];
    int32_t fb_amax[kMaxRows];
    int32_t n_fallback;
    int32_t bar_ok;
    // phase 2, the truncated row being finished
    float fin_m;
    int32_t fin_amax;
    uint32_t fin_flags;
    uint32_t fin_over;
    int32_t n_sel;
    unsigned long long fin_tinc;  // tokens missing from every list lie below it
    // CTA-wide scratch for the exact fallback
    uint32_t hcnt[256];
    unsigned long long hmass[256];
    unsigned long long scan_w[kW];
    int32_t red_i[kW];
    float red_f[kW];
    GTop2 red_g[kW];
    unsigned long long sel_prefix;  // state of the fallback select
    unsigned long long sel_wabove;
    unsigned long long sel_target;
    int32_t sel_idx;
    int32_t sel_found;
};

constexpr size_t kSharedHead = (sizeof(ColShared) + 127) & ~size_t(127);
constexpr size_t kWarpBytes = size_t(kSlotBytes) + size_t(kBufCap) * 8;
constexpr size_t kSmemBytes = kSharedHead + kW * kWarpBytes;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// phase 2 reuses the warps' slots: the records' lists, then the gathered tokens
static_assert(size_t(kMaxUnits) * (kCandCap * 8 + 7 * 4) + size_t(kSelCap) * 20 <= kW * kWarpBytes,
              "phase-2 area");

__device__ __forceinline__ RowParams as_row_params(const RowInfo& ri)
{
    RowParams rp;
    rp.T = ri.T;
    rp.Te = ri.Te;
    rp.invT = ri.invT;
    rp.k = ri.k;
    rp.p = ri.p;
    rp.minp = ri.minp;
    rp.pres = 0.0f;
    rp.freq = 0.0f;
    rp.rep = 1.0f;
    rp.lrow = ri.lrow;
    rp.hlo = rp.hhi = 0;
    rp.stream = ri.stream;
    rp.status = ri.status;
    rp.greedy = ri.greedy;
    rp.do_topk = ri.do_topk;
    rp.do_topp = ri.do_topp;
    rp.do_minp = ri.do_minp;
    rp.want_out = 0;
    rp.has_hist = 0;
    rp.plain_single = ri.cls == kClsPlain;
    rp.key_lo = ri.key_lo;
    rp.key_hi = ri.key_hi;
    rp.off_lo = ri.off_lo;
    rp.off_hi = ri.off_hi;
    return rp;
}

// Composite sort word of an fp32 value and its token.
__device__ __forceinline__ unsigned long long comp_of(float x, int v) { return cand_word(f2key(x), v); }

// ---------------------------------------------------------------- warp helpers
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
        v = o > v ? o : v;
    }
    return v;
}

// Sort n <= kBufCap words in warp-private shared memory, descending (bitonic,
// padded to a power of two with zeros; the array must hold that many words).
__device__ __forceinline__ void warp_sort_smem_desc(unsigned long long* a, int n)
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

// Sort n <= kSelCap words in shared memory, descending, with the whole CTA: each
// word's rank is the number of words above it (words are distinct), found by
// kT / n threads per word, then the words are scattered. rank[] and out[] hold n.
__device__ __forceinline__ void cta_rank_sort_desc(const unsigned long long* in, int n, uint32_t* rank,
                                                   unsigned long long* out)
{
    const int tid = threadIdx.x;
    for (int i = tid; i < n; i += kT) rank[i] = 0u;
    __syncthreads();
    const int per = n > 0 ? max(1, kT / n) : 1;  // threads per word
    const int chunk = (n + per - 1) / per;
    for (int t = tid; t < n * per; t += kT) {
        const int i = t % n, c = t / n;
        const unsigned long long x = in[i];
        uint32_t above = 0;
        const int j1 = min(n, (c + 1) * chunk);
        for (int j = c * chunk; j < j1; ++j) above += in[j] > x ? 1u : 0u;
        if (above) atomicAdd(&rank[i], above);
    }
    __syncthreads();
    for (int i = tid; i < n; i += kT) out[rank[i]] = in[i];
    __syncthreads();
}

}  // namespace col
}  // namespace dst

namespace dst {
namespace col {

// ---------------------------------------------------------------- CTA-wide helpers (fallback)
__device__ __forceinline__ unsigned long long cta_suffix_scan(unsigned long long v, ColShared& sh)
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

__device__ __forceinline__ int cta_excl_scan(int v, int& total, ColShared& sh)
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

// Exact kept-prefix selection over a whole row, streamed from global memory by
// one CTA: the first token whose inclusive weight (count, or fixed-point mass)
// reaches `target` closes the prefix. Tokens outside the domain prefix weigh 0.
template <typename InT>
__device__ void cta_select(ColShared& sh, const KernelParams& kp, const RowInfo& ri, int V,
                           bool mass_mode, bool dom, uint32_t dkey, int didx, float m,
                           unsigned long long count_target, uint32_t& out_key, int& out_idx)
{
    const int tid = threadIdx.x;
    if (tid == 0) {
        sh.sel_prefix = 0;
        sh.sel_wabove = 0;
        sh.sel_target = count_target;
    }
    __syncthreads();
    uint32_t pbits = 0;
    unsigned long long tie_J = 1;
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
    {
        const unsigned long long wt = mass_mode ? mass_q(key2f(K), m, ri.invT) : 1ull;
        tie_J = (sh.sel_target - sh.sel_wabove + wt - 1) / wt;
    }
    // the tie_J-th token (index order) holding key K
    int base = 0;
    int found = -1;
    for (int v0 = 0; v0 < V; v0 += kT) {
        const int v = v0 + tid;
        int c = 0;
        if (v < V) {
            const float x = row_x<InT>(kp, ri.lrow, v);
            const uint32_t key = f2key(x);
            c = (key == K && (!dom || in_prefix(key, v, dkey, didx))) ? 1 : 0;
        }
        int total = 0;
        const int excl = cta_excl_scan(c, total, sh);
        if (c && (unsigned long long)(base + excl + 1) == tie_J) sh.sel_idx = v;
        base += total;
        if ((unsigned long long)base >= tie_J) break;
    }
    __syncthreads();
    (void)found;
    out_key = K;
    out_idx = sh.sel_idx;
    __syncthreads();
}

// Exact finish of one row by the whole CTA (rows the candidates could not settle).
template <typename InT>
__device__ void cta_exact_row(ColShared& sh, const ColParams& P, int r, const RowInfo ri, float m,
                              int amax)
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
        const double th = double(m) + double(ri.Te) * log(double(ri.minp));
        float f = float(th);
        if (double(f) < th) f = nextafterf(f, INFINITY);
        xthr = f;
    }
    const RowParams rp = as_row_params(ri);
    GumbelAcc g;
    gumbel_init(g);
    for (int v = tid; v < V; v += kT) {
        const float x = row_x<InT>(kp, ri.lrow, v);
        if (!(x > -INFINITY)) continue;
        if (hb && !in_prefix(f2key(x), v, bk, bi)) continue;
        if (ri.do_minp && !(x >= xthr)) continue;
        gumbel_visit(g, rp, v, x);
    }
    top2_warp_reduce(g.t);
    if (lane == 0) sh.red_g[wid] = g.t;
    __syncthreads();
    if (tid == 0) {
        GTop2 t;
        t.a = grec_empty();
        t.b = grec_empty();
        for (int w = 0; w < kW; ++w) {
            top2_insert(t, sh.red_g[w].a);
            top2_insert(t, sh.red_g[w].b);
        }
        kp.out_tokens[r] = ri.greedy ? amax : settle_top2(t, ri.T);
        if (kp.out_status) kp.out_status[r] = kRowOk;
    }
    __syncthreads();
}

}  // namespace col
}  // namespace dst
