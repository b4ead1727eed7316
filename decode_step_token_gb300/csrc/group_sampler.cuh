// group_sampler.cuh -- the fork-group sampler kernel for large batches (sm_103a).
//
// A persistent grid of thread-block clusters walks the batch in chunks of output
// rows. Inside a chunk, consecutive output rows that read the same logits row
// (forks: n samples of one prompt, each with its own Philox stream) form a
// group; the cluster stages that logits row once -- each of its C CTAs copies one
// contiguous part into shared memory with bulk (TMA-engine) copies -- and serves
// every fork of the group from shared memory. Per group:
//
//   P1  each CTA: its part's max / argmax / non-finite flags, each thread's
//       maximum (the thread maxima bound the top-k / top-p cut from below), the
//       softmax mass sum per temperature that needs it, and the Gumbel-max pick
//       of forks that truncate nothing
//   R1  leader CTA: row max and status, picks of greedy and plain forks, and per
//       truncating fork a provable lower bound tau of its kept set: the min-p
//       threshold, the value reached by k thread maxima (top-k), or the value
//       above which the thread maxima alone carry p of the mass (top-p)
//   P2  each CTA lists its tokens at or above the smallest tau
//   R2  leader CTA: sorts the list by (value desc, index asc), cuts top-k,
//       top-p and min-p per fork in the kept order, and takes the Gumbel-max
//       pick over the kept tokens (fp32 scores, best two settled in double)
//   P3  optional fp32 probs / logprobs of every fork, from shared memory
//
// A fork whose kept set the list cannot settle (no bound, or the list overflowed)
// takes the exact path: a cluster-wide radix select by count or by fixed-point
// softmax mass over the staged row, then a Gumbel pass over the kept prefix.
// Rows with penalties are never grouped (their penalised logits differ).
//
// Stage definitions: xbrilliance.ai note on sampling cost, section
// "解码一步里采样做什么"; the Gumbel-max pick: dev.to, "SGLang's +75% sampler
// speedup skips Qwen3 chat requests", section "Nine lines, and exactly one call site".
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "row_sampler.cuh"

namespace dst {
namespace grp {

constexpr int kT = 256;
constexpr int kW = kT / 32;
constexpr int kMaxForks = 8;     // output rows per group
constexpr int kMaxParts = 8;     // CTAs per cluster
constexpr int kChunks = 4;       // bulk copies per part
constexpr uint32_t kPolls = 1u << 24;

enum : int32_t {
    kKindDone = 0,   // token known after R1 (error, greedy without outputs, plain)
    kKindList = 1,   // the cut comes from the candidate list
    kKindExact = 2,  // the cut comes from the exact path
    kKindAll = 3,    // kept set = every finite token: token and mass known after R1
    kKindPick = 4,   // the cut is known: the pick pass takes the token and kept mass
};

struct GroupParams {
    KernelParams k;
    int32_t n_rows;
    int32_t chunk;      // output rows per work chunk; groups never span chunks
    int32_t n_chunks;
    int32_t group;      // 1: rows may share a staged logits row; 0: one row per group
    int32_t slice_len;  // elements per CTA, a multiple of 16
    int32_t list_cap;   // merged candidates the leader sorts (a power of two)
    int32_t part_cap;   // candidates one CTA may list
    uint32_t off_list;  // dynamic shared memory layout, bytes
    uint32_t off_cand;
    uint32_t off_cnt;
    uint32_t off_stage;
    uint32_t* work;     // [2] chunks handed out past the first one per cluster, clusters done;
                        // zero between launches (the last cluster to finish clears them)
};

struct alignas(8) ForkOut {  // leader's result for one fork, copied to every CTA
    int32_t status;
    int32_t token;
    int32_t kind;
    int32_t has_bound;
    float xthr;    // min-p threshold, -inf when off
    float tau;     // lower bound of the kept set (kKindCand)
    float lnz;     // ln of the kept mass relative to exp((x - m) / Te)
    uint32_t bkey; // last kept token (value key, index) when has_bound
    int32_t bidx;
    int32_t listed;  // every kept token is in the candidate lists
};

struct alignas(8) GPartial {  // one CTA's summary of its part
    float mx;
    int32_t amax;
    uint32_t flags;
    uint32_t ncand;
    double z[kMaxForks];      // per fork slot: sum of exp((x - mx) / Te) over the part
    GTop2 g[kMaxForks];       // the part's best two Gumbel scores per fork
    double zk[kMaxForks];     // pick pass: kept mass per fork, relative to the row max
};

struct alignas(8) GBcast {  // group-wide leader results
    float m;
    int32_t amax;
    int32_t status;   // base-row status (non-finite, all -inf, timeout)
    float tau_all;    // smallest tau over the forks that gather
    int32_t gather;   // some fork needs the candidate list
    int32_t exact;    // some fork takes the exact path
    int32_t out;      // the call writes probs / logprobs
    int32_t pick;     // some fork needs the pick pass
    ForkOut f[kMaxForks];
};

struct alignas(8) SelState {  // exact path: radix select state
    uint32_t prefix;
    uint32_t pbits;
    unsigned long long w_above;
    unsigned long long target;
    int32_t tie_cta;
    int32_t tie_j;
    int32_t bidx;
    int32_t pad;
};

struct alignas(16) GShared {
    uint64_t mbar[kChunks];
    int32_t next_chunk[2]; // the cluster's next chunk, by iteration parity (written by the leader)
    uint32_t phase;        // parity of the next wait on mbar[]
    int32_t n_forks;
    int32_t r0;
    int32_t lrow;
    int32_t nch, hb, head_end, tail_begin;
    int32_t ncand;
    int32_t zslots;        // distinct Z slots
    int32_t zslot_fork[kMaxForks];  // fork that defines each slot (its Te)
    RowParams rp[kMaxForks];
    int32_t zslot_of[kMaxForks];
    double zrow[kMaxForks];        // leader: the row's mass per fork, relative to m
    double lnmp[kMaxForks];        // Te * ln(min_p) per fork
    GPartial part;
    GBcast bc;
    SelState sel;
    float red_f[kW];
    int32_t red_i[kW];
    uint32_t red_u[kW];
    double red_d[kW];
    unsigned long long red_q[kW];
    GTop2 red_g[kW];
    uint32_t tmax[kT];             // this CTA's thread maxima (value keys)
    uint32_t hcnt[256];            // exact path histograms
    unsigned long long hmass[256];
};

// ------------------------------------------------------------------ staged part
struct Part {
    const unsigned char* stage;  // element i at byte hb + i * esize
    const uint16_t* cnt;         // history counts (bf16 rows with penalties), else null
    int n;                       // elements in the part
    int hoff;                    // head pad in elements
    int v0;                      // first token
};

template <typename InT>
__device__ __forceinline__ float part_x(const Part& pt, const RowParams& rp, int i)
{
    const unsigned char* p = pt.stage + (pt.hoff + i) * int(sizeof(InT));
    float x;
    if (sizeof(InT) == 4) x = *reinterpret_cast<const float*>(p);
    else x = __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(p)) << 16);
    if (sizeof(InT) == 2 && pt.cnt) {
        const uint32_t c = pt.cnt[i];
        if (c) x = penalize(x, c, rp);
    }
    return x;
}

// Visit every element of the part as (token, fp32 logit), 16-byte vectors per thread.
template <typename InT, typename F>
__device__ __forceinline__ void part_for_each(const Part& pt, const RowParams& rp, F&& f)
{
    constexpr int EPV = ElemTraits<InT>::kPerVec;
    const int nvec = (pt.hoff + pt.n + EPV - 1) / EPV;
    const uint4* vec = reinterpret_cast<const uint4*>(pt.stage);
    for (int j = threadIdx.x; j < nvec; j += kT) {
        const uint4 raw = vec[j];
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const int i = j * EPV + e - pt.hoff;
            if (i < 0 || i >= pt.n) continue;
            float x = ElemTraits<InT>::get(raw, e);
            if (sizeof(InT) == 2 && pt.cnt) {
                const uint32_t c = pt.cnt[i];
                if (c) x = penalize(x, c, rp);
            }
            f(pt.v0 + i, x);
        }
    }
}

// Maximum of a 16-byte vector of logits (NaN ignored), whether it holds a NaN, and
// the first position holding a given value.
template <typename InT>
struct VecMax;

template <>
struct VecMax<uint16_t> {
    static constexpr int E = 8;
    __device__ static __forceinline__ float vmax(const uint4& r, bool& nan)
    {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
        const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
        const __nv_bfloat162 mx = __hmax2(__hmax2(a, b), __hmax2(c, d));             // NaN ignored
        const __nv_bfloat162 mn = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));  // NaN kept
        const float n0 = __low2float(mn), n1 = __high2float(mn);
        nan = (n0 != n0) || (n1 != n1);
        return fmaxf(__low2float(mx), __high2float(mx));
    }
};

template <>
struct VecMax<float> {
    static constexpr int E = 4;
    __device__ static __forceinline__ float vmax(const uint4& r, bool& nan)
    {
        const float a = __uint_as_float(r.x), b = __uint_as_float(r.y);
        const float c = __uint_as_float(r.z), d = __uint_as_float(r.w);
        nan = (a != a) || (b != b) || (c != c) || (d != d);
        return fmaxf(fmaxf(a, b), fmaxf(c, d));
    }
};

template <typename InT>
__device__ __forceinline__ int vec_first(const uint4& r, float v)
{
    int pos = VecMax<InT>::E - 1;
#pragma unroll
    for (int e = VecMax<InT>::E - 1; e >= 0; --e)
        if (ElemTraits<InT>::get(r, e) == v) pos = e;
    return pos;
}

// ------------------------------------------------------------------ register sort
template <typename T>
__device__ __forceinline__ T shfl_xor_any(T v, int m)
{
    return __shfl_xor_sync(0xffffffffu, v, m);
}

// Bitonic sort, descending, of PER * kT words: word i = q * kT + tid sits in v[q] of
// thread tid. Pairs inside one thread swap in registers, pairs inside one warp
// through shuffles, the rest through `xs` (PER * kT words of shared memory).
template <typename T, int PER>
__device__ __forceinline__ void reg_sort_desc(T (&v)[PER], T* xs)
{
    const int tid = threadIdx.x;
    constexpr int N = PER * kT;
#pragma unroll 1
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll 1
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= kT) {
                const int qs = stride / kT;
#pragma unroll
                for (int q = 0; q < PER; ++q) {
#pragma unroll
                    for (int p = q + 1; p < PER; ++p) {
                        if ((q ^ p) != qs) continue;
                        const bool desc = ((q * kT + tid) & size) == 0;
                        const T a = v[q], b = v[p];
                        const bool sw = desc ? (a < b) : (a > b);
                        v[q] = sw ? b : a;
                        v[p] = sw ? a : b;
                    }
                }
            } else if (stride >= 32) {
                __syncthreads();
#pragma unroll
                for (int q = 0; q < PER; ++q) xs[q * kT + tid] = v[q];
                __syncthreads();
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    const int i = q * kT + tid;
                    const T o = xs[i ^ stride];
                    const bool keep_max = ((i & stride) == 0) == ((i & size) == 0);
                    v[q] = keep_max ? (v[q] > o ? v[q] : o) : (v[q] < o ? v[q] : o);
                }
            } else {
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    const int i = q * kT + tid;
                    const T o = shfl_xor_any(v[q], stride);
                    const bool keep_max = ((i & stride) == 0) == ((i & size) == 0);
                    v[q] = keep_max ? (v[q] > o ? v[q] : o) : (v[q] < o ? v[q] : o);
                }
            }
        }
    }
    __syncthreads();
}

// Sort n words of `a` (shared memory) descending: n is padded with zero words up to
// a power of two of at least kT, which `a` must hold.
template <typename T>
__device__ __noinline__ void sort_desc(T* a, int n)
{
    int np2 = kT;
    while (np2 < n) np2 <<= 1;
    for (int i = n + int(threadIdx.x); i < np2; i += kT) a[i] = T(0);
    __syncthreads();
    auto run = [&](auto per_tag) {
        constexpr int PER = decltype(per_tag)::value;
        T v[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) v[q] = a[q * kT + threadIdx.x];
        reg_sort_desc<T, PER>(v, a);
#pragma unroll
        for (int q = 0; q < PER; ++q) a[q * kT + threadIdx.x] = v[q];
        __syncthreads();
    };
    switch (np2 / kT) {
        case 1: run(std::integral_constant<int, 1>()); break;
        case 2: run(std::integral_constant<int, 2>()); break;
        case 4: run(std::integral_constant<int, 4>()); break;
        case 8: run(std::integral_constant<int, 8>()); break;
        default: run(std::integral_constant<int, 16>()); break;
    }
}

// ------------------------------------------------------------------ block helpers
__device__ __forceinline__ double block_sum_f64(double v, GShared& sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if (lane == 0) sh.red_d[wid] = v;
    __syncthreads();
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < kW; ++w) t += sh.red_d[w];
    return t;
}

// Inclusive prefix sum (index order) of one double per thread over the block.
__device__ __forceinline__ double block_incl_scan_f64(double v, GShared& sh, double& total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    double s = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double o = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += o;
    }
    __syncthreads();
    if (lane == 31) sh.red_d[wid] = s;
    __syncthreads();
    double before = 0.0, tot = 0.0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
        if (w < wid) before += sh.red_d[w];
        tot += sh.red_d[w];
    }
    total = tot;
    return before + s;
}

__device__ __forceinline__ int block_sum_i32(int v, GShared& sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if (lane == 0) sh.red_i[wid] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) t += sh.red_i[w];
    return t;
}

// Sort n (a power of two, <= capacity) words in shared memory, descending.
__device__ __forceinline__ void block_sort_desc(unsigned long long* a, int n)
{
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = threadIdx.x; t < (n >> 1); t += kT) {
                const int lo = ((t & ~(stride - 1)) << 1) | (t & (stride - 1));
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

}  // namespace grp
}  // namespace dst
