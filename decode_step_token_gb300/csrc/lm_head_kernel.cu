// lm_head_kernel.cu -- the LM-head GEMM that produces a decode step's logits,
// logits[r, v] = bf16(sum_k hidden[r, k] * weight[v, k]), on the fifth-generation
// tensor cores (tcgen05.mma, fp32 accumulators in tensor memory) with both
// operands staged by the TMA engine, chained to the sampler by programmatic
// dependent launch.
//
// The xbrilliance.ai note on sampling cost (section "解码一步里采样做什么")
// has the LM head compute the [num_seqs, vocab_size] logits as
// matmul(hidden_states, embedding.t()) and hand them to Sampler.forward.
//
// A decode batch is skinny (tens of rows against a vocabulary of 10^5), so the
// product is taken transposed: a tile is 128 weight rows (operand A, M = 128)
// against every hidden row (operand B, N = rows rounded up to 16), K in stages
// of 64 (one 128-byte swizzled row per operand row). The weight streams from
// HBM once per step; the hidden rows are re-read from L2. The kernel is
// persistent (one CTA per SM, tiles dealt round-robin) with warp roles:
//   warp 0     one thread issues the TMA loads of a ring of stages;
//   warp 1     owns the tensor memory (two accumulators of N columns) and one
//              thread issues the MMAs, freeing a stage with tcgen05.commit;
//   warps 2-5  the epilogue: each reads its 32 tensor-memory lanes (tile rows)
//              with tcgen05.ld, rounds to bf16 and stores the logits, while the
//              MMAs of the next tile fill the other accumulator.
// Every wait is bounded in time (global timer); a CTA whose wait gives up
// counts itself in the handle's statistics and leaves its logits unwritten.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "ptx.cuh"

namespace dst {
namespace lmh {

constexpr int kBM = 128;                 // weight rows per tile (MMA M)
constexpr int kBK = 64;                  // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUK = 16;                  // K of one tcgen05.mma (kind::f16)
constexpr int kThreads = 192;            // six warps (roles above)
constexpr int kMaxStages = 8;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB per stage
constexpr uint64_t kWaitNs = 2000000000ull;  // a CTA's waits give up 2 s after it starts
constexpr uint64_t kDrainNs = 1000000000ull; // and its final drains 1 s after that
constexpr size_t kBarBytes = 256;        // mbarriers, the tensor-memory address, a flag
constexpr size_t kSmemMax = 227 * 1024;

struct Params {
    CUtensorMap tw;      // weight [V, K] bf16: box 64 x 128, 128-byte swizzle
    CUtensorMap th;      // hidden [n, K] bf16: box 64 x NT, 128-byte swizzle
    uint16_t* logits;    // [n, ldl] bf16
    int64_t ldl;
    int n, NT, V;
    int tiles, kchunks, stages;
    uint32_t tmem_cols;  // a power of two >= 2 * NT
    unsigned long long* timeouts;  // CTAs whose wait gave up (may be NULL)
};

// Shared-memory matrix descriptor of a K-major bf16 tile in the 128-byte
// swizzled layout written by the TMA engine: rows of 128 bytes, 8-row atoms
// 1024 bytes apart (stride byte offset), the leading byte offset unused.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr)
{
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint64_t now_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity, giving up at `deadline`
// (global timer, ns); returns success.
__device__ __forceinline__ bool wait_until(uint64_t* bar, uint32_t parity, uint64_t deadline)
{
    for (uint32_t i = 0; i < (1u << 30); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && now_ns() > deadline) return false;
    }
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) lm_head_kernel(const __grid_constant__ Params P)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // operand stages on 1024-byte boundaries (the swizzle pattern repeats every 1024 bytes)
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int S = P.stages;
    const uint32_t b_bytes = uint32_t(P.NT) * kBK * 2;
    unsigned char* sa = smem;
    unsigned char* sb = smem + size_t(S) * kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sb + size_t(S) * b_bytes);
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;  // [2] an accumulator is complete
    uint64_t* tempty = tfull + 2;          // [2] an accumulator has been read
    uint64_t* drained = tempty + 2;        // every MMA of the CTA has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drained + 1);
    int* gave_up = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t deadline = now_ns() + kWaitNs;
    // the sampler may launch now: it waits for this grid before it reads the logits
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(drained, 1);
        *gave_up = 0;
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tw)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.th)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(P.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int G = int(gridDim.x), b = int(blockIdx.x);
    const int my_tiles = P.tiles > b ? (P.tiles - 1 - b) / G + 1 : 0;

    if (warp == 0) {
        if (lane == 0) {  // TMA producer
            int it = 0;
            bool ok = true;
            for (int t = 0; ok && t < my_tiles; ++t) {
                const int row0 = (b + t * G) * kBM;
                for (int kc = 0; kc < P.kchunks; ++kc) {
                    const int s = it % S;
                    const uint32_t use = uint32_t(it / S);
                    if (!wait_until(&empty[s], (use & 1u) ^ 1u, deadline)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], kABytes + b_bytes);
                    tma_load_2d(smem_addr(sa + size_t(s) * kABytes), &P.tw, kc * kBK, row0, smem_addr(&full[s]));
                    tma_load_2d(smem_addr(sb + size_t(s) * b_bytes), &P.th, kc * kBK, 0, smem_addr(&full[s]));
                    ++it;
                }
            }
            if (!ok) *gave_up = 1;
            // the last copies issued land before the CTA may exit
            for (int j = it > S ? it - S : 0; j < it; ++j)
                wait_until(&full[j % S], uint32_t(j / S) & 1u, deadline + kDrainNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t idesc = idesc_bf16(kBM, P.NT);
            int it = 0;
            bool ok = true;
            for (int t = 0; ok && t < my_tiles; ++t) {
                const int acc = t & 1;
                const uint32_t use = uint32_t(t >> 1);
                if (!wait_until(&tempty[acc], (use & 1u) ^ 1u, deadline)) {
                    ok = false;
                    break;
                }
                fence_after_sync();
                const uint32_t d = tmem + uint32_t(acc * P.NT);
                for (int kc = 0; kc < P.kchunks; ++kc) {
                    const int s = it % S;
                    if (!wait_until(&full[s], uint32_t(it / S) & 1u, deadline)) {
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    const uint64_t da = desc_sw128(smem_addr(sa + size_t(s) * kABytes));
                    const uint64_t db = desc_sw128(smem_addr(sb + size_t(s) * b_bytes));
#pragma unroll
                    for (int k = 0; k < kBK / kUK; ++k)  // +32 bytes per K step inside the 128-byte rows
                        mma_bf16(d, da + uint64_t(2 * k), db + uint64_t(2 * k), idesc, uint32_t(kc | k));
                    mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
                    ++it;
                }
                if (ok) mma_commit(&tfull[acc]);
            }
            if (!ok) *gave_up = 1;
            mma_commit(drained);
            wait_until(drained, 0, deadline + kDrainNs);
        }
    } else {  // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
        const int q = warp & 3;
        bool ok = true;
        for (int t = 0; t < my_tiles; ++t) {
            const int acc = t & 1;
            if (!wait_until(&tfull[acc], uint32_t(t >> 1) & 1u, deadline)) {
                ok = false;
                break;
            }
            fence_after_sync();
            const int v = (b + t * G) * kBM + q * 32 + lane;
            const uint32_t base = tmem + (uint32_t(q * 32) << 16) + uint32_t(acc * P.NT);
            for (int c0 = 0; c0 < P.NT; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(base + uint32_t(c0), r);
                if (v < P.V) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < P.n)
                            P.logits[size_t(c0 + j) * size_t(P.ldl) + size_t(v)] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[j])));
                }
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        if (!ok && lane == 0) *gave_up = 1;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P.tmem_cols) : "memory");
    if (tid == 0 && *gave_up && P.timeouts) atomicAdd(P.timeouts, 1ull);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor map over rows x cols (row stride `ld` elements), box 64 x box_rows,
// 128-byte swizzle; elements outside the tensor read as zero.
bool encode(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(ld) * 2u};
    const cuuint32_t box[2] = {cuuint32_t(kBK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace lmh

bool lm_head_plan(int64_t rows, int64_t vocab, int64_t hidden_dim, int sms, LmHeadPlan* plan)
{
    if (rows < 1 || rows > kLmHeadMaxRows || vocab < 1 || hidden_dim < 1 || sms < 1) return false;
    const int NT = int((rows + 15) / 16 * 16);
    const size_t stage = lmh::kABytes + size_t(NT) * lmh::kBK * 2;
    const int stages = int(std::min<size_t>(lmh::kMaxStages, (lmh::kSmemMax - 1024 - lmh::kBarBytes) / stage));
    if (stages < 2) return false;
    uint32_t cols = 32;
    while (cols < uint32_t(2 * NT)) cols <<= 1;
    plan->NT = NT;
    plan->stages = stages;
    plan->tmem_cols = cols;
    plan->tiles = int((vocab + lmh::kBM - 1) / lmh::kBM);
    plan->kchunks = int((hidden_dim + lmh::kBK - 1) / lmh::kBK);
    plan->ctas = std::min(sms, plan->tiles);
    plan->smem = 1024 + size_t(stages) * stage + lmh::kBarBytes;
    return true;
}

int lm_head_prepare(size_t smem)
{
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&lmh::lm_head_kernel),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

int lm_head_launch(const sampler_lm_head_t* g, void* logits, int64_t ldl, int64_t rows, int64_t vocab,
                   const LmHeadPlan& plan, unsigned long long* timeouts, cudaStream_t stream)
{
    lmh::Params p;
    std::memset(&p, 0, sizeof p);
    if (!lmh::encode(&p.tw, g->weight, vocab, g->hidden_dim, g->weight_stride, lmh::kBM) ||
        !lmh::encode(&p.th, g->hidden, rows, g->hidden_dim, g->hidden_stride, plan.NT))
        return SAMPLER_ERR_CUDA;
    p.logits = static_cast<uint16_t*>(logits);
    p.ldl = ldl;
    p.n = int(rows);
    p.NT = plan.NT;
    p.V = int(vocab);
    p.tiles = plan.tiles;
    p.kchunks = plan.kchunks;
    p.stages = plan.stages;
    p.tmem_cols = plan.tmem_cols;
    p.timeouts = timeouts;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(unsigned(plan.ctas));
    cfg.blockDim = dim3(lmh::kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    void* args[] = {&p};
    if (cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&lmh::lm_head_kernel), args) != cudaSuccess)
        return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

}  // namespace dst
