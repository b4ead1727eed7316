// sampler_api.cu -- the C ABI of libsampler.so (declared in include/sampler.h):
// argument checks, launch geometry and the cluster launch of the row kernel,
// plus the host-buffer entry that stages through the handle's device buffers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "colsplit_kernel.cuh"
#include "group_sampler_kernel.cuh"
#include "row_sampler_kernel.cuh"
#include "sampler.h"

namespace {

constexpr int64_t kMaxVocabLimit = 262144;  // a row always fits one cluster's shared memory
constexpr int kMaxSmem = 227 * 1024;
constexpr int kNumStats = 4;

struct Geometry {
    int cluster;    // CTAs per row
    int slice;      // elements per CTA
    size_t smem;    // dynamic shared memory per CTA
};

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

Geometry geometry(int64_t V, int esize, bool pen)
{
    Geometry g;
    g.cluster = int(std::min<int64_t>(dst::kMaxCluster, std::max<int64_t>(1, (V + 16383) / 16384)));
    int64_t l = (V + g.cluster - 1) / g.cluster;
    l = (l + 7) & ~int64_t(7);
    g.slice = int(l);
    g.smem = align16(sizeof(dst::Shared)) + (pen ? align16(size_t(l) * 2 + 4) : 0) +
             align16(size_t(l) * esize + 32);
    return g;
}

template <typename InT, bool kPen>
void* kernel_ptr()
{
    return reinterpret_cast<void*>(&dst::row_sampler_kernel<InT, kPen>);
}

void* pick_kernel(int dtype, bool pen)
{
    if (dtype == SAMPLER_DTYPE_BF16) return pen ? kernel_ptr<uint16_t, true>() : kernel_ptr<uint16_t, false>();
    return pen ? kernel_ptr<float, true>() : kernel_ptr<float, false>();
}

int kernel_slot(int dtype, bool pen) { return (dtype == SAMPLER_DTYPE_BF16 ? 2 : 0) + (pen ? 1 : 0); }

}  // namespace

struct sampler_s {
    int device;
    int num_sms;
    int64_t max_rows, max_vocab, max_history;
    uint32_t flags;
    size_t smem_set[4];  // dynamic shared memory already granted per kernel variant
    size_t col_smem_set[2];
    size_t grp_smem_set[4];
    size_t grp_occ_smem[4];  // shared memory of the cached cluster occupancy below
    int grp_occ[4];          // co-resident clusters of the fork-group kernel
    // workspace of the unit-split path: per-(row, unit) records and the per-row counters
    dst::col::ColRec* col_rec;
    dst::col::RowSync* col_bar;
    unsigned long long* stats;  // device counters (diagnostics)
    int col_rows;
    int64_t col_units;  // records in col_rec
    // staging for sampler_sample_host
    unsigned char* stage_base;
    size_t stage_bytes;
};

namespace {

struct ColGeometry {
    int gc;         // units per row
    int w;          // elements per unit
    int64_t units;  // n_rows * gc
    int grid;       // CTAs
};
bool col_eligible(sampler_t h, const sampler_args_t* a, ColGeometry* g);
int launch_col(sampler_t h, const sampler_args_t* a, const ColGeometry& g, cudaStream_t stream);

// ---------------------------------------------------------------- fork-group kernel
constexpr size_t kTwoPerSm = 113 * 1024;  // dynamic shared memory that lets two CTAs share an SM

struct GroupGeometry {
    int parts;       // CTAs per cluster
    int slice;       // elements per CTA
    int list_cap, part_cap;
    uint32_t off_list, off_cand, off_cnt, off_stage;
    size_t smem;
};

// Parts of at most 64 KB each (up to eight), then the largest candidate lists that
// keep two CTAs per SM; fp32 rows with penalties reuse the count table's space for
// the lists (the counts are folded into the staged row before any list exists).
bool group_geometry(int64_t V, int esize, bool pen, GroupGeometry* g)
{
    const int64_t parts = std::min<int64_t>(dst::grp::kMaxParts, std::max<int64_t>(1, (V * esize + 65535) / 65536));
    int64_t l = (V + parts - 1) / parts;
    l = (l + 15) & ~int64_t(15);
    g->parts = int(parts);
    g->slice = int(l);
    const size_t head = (sizeof(dst::grp::GShared) + 127) & ~size_t(127);
    const size_t stage = align16(size_t(l) * esize + 32);
    const size_t cnt = pen ? align16(size_t(l) * 2 + 16) : 0;
    for (int pass = 0; pass < 2; ++pass) {
        const size_t limit = pass == 0 ? kTwoPerSm : size_t(kMaxSmem) - 1024;
        for (int cap = 4096; cap >= (pass == 0 ? 1024 : 256); cap >>= 1) {
            // the leader also bins the row's thread maxima (4 x 256 words) in the list area
            if (size_t(cap) * 8 < 4096) break;
            const int pcap = std::min(cap, 1024);
            const size_t lists = size_t(cap) * 8 + size_t(pcap) * 8;
            const bool alias = pen && esize == 4;
            const size_t region = alias ? std::max(cnt, lists) : lists + cnt;
            const size_t total = head + region + stage;
            if (total > limit) continue;
            g->list_cap = cap;
            g->part_cap = pcap;
            g->off_list = uint32_t(head);
            g->off_cand = uint32_t(head + size_t(cap) * 8);
            g->off_cnt = uint32_t(alias ? head : head + lists);
            g->off_stage = uint32_t(head + region);
            g->smem = total;
            return true;
        }
    }
    return false;
}

template <typename InT, bool kPen>
void* grp_kernel_ptr()
{
    return reinterpret_cast<void*>(&dst::grp::group_kernel<InT, kPen>);
}

void* grp_pick(int dtype, bool pen)
{
    if (dtype == SAMPLER_DTYPE_BF16) return pen ? grp_kernel_ptr<uint16_t, true>() : grp_kernel_ptr<uint16_t, false>();
    return pen ? grp_kernel_ptr<float, true>() : grp_kernel_ptr<float, false>();
}

int launch_group(sampler_t h, const sampler_args_t* a, const GroupGeometry& gg, cudaStream_t stream)
{
    const bool pen = a->hist_offsets != nullptr;
    void* fn = grp_pick(a->dtype, pen);
    const int slot = kernel_slot(a->dtype, pen);
    if (h->grp_smem_set[slot] < gg.smem) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(gg.smem)) != cudaSuccess)
            return SAMPLER_ERR_CUDA;
        h->grp_smem_set[slot] = gg.smem;
    }
    dst::grp::GroupParams p;
    std::memset(&p, 0, sizeof p);
    dst::KernelParams& k = p.k;
    k.logits = a->logits;
    k.vocab = a->vocab;
    k.row_stride = a->row_stride;
    k.n_logit_rows = a->n_logit_rows > 0 ? a->n_logit_rows : a->n_rows;
    k.logit_row = a->logit_row;
    k.temperature = a->temperature;
    k.top_k = a->top_k;
    k.top_p = a->top_p;
    k.min_p = a->min_p;
    k.presence = a->presence_penalty;
    k.frequency = a->frequency_penalty;
    k.repetition = a->repetition_penalty;
    k.seed = a->seed;
    k.has_seed = a->has_seed;
    k.stream_id = a->stream_id;
    k.hist_offsets = a->hist_offsets;
    k.hist_ids = a->hist_ids;
    k.global_seed = a->global_seed;
    k.philox_offset = a->philox_offset;
    k.philox_offset_dev = a->philox_offset_dev;
    k.out_tokens = a->out_tokens;
    k.out_probs = a->out_probs;
    k.out_logprobs = a->out_logprobs;
    k.out_status = a->out_status;
    k.slice_len = gg.slice;
    p.n_rows = int(a->n_rows);
    p.group = (a->logit_row != nullptr && !pen) ? 1 : 0;
    p.chunk = p.group ? dst::grp::kMaxForks : 1;
    p.n_chunks = int((a->n_rows + p.chunk - 1) / p.chunk);
    p.slice_len = gg.slice;
    p.list_cap = gg.list_cap;
    p.part_cap = gg.part_cap;
    p.off_list = gg.off_list;
    p.off_cand = gg.off_cand;
    p.off_cnt = gg.off_cnt;
    p.off_stage = gg.off_stage;

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.blockDim = dim3(dst::grp::kT, 1, 1);
    cfg.dynamicSmemBytes = gg.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(gg.parts);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a persistent grid: as many clusters as fit at once, never more than chunks
    if (h->grp_occ_smem[slot] != gg.smem || h->grp_occ[slot] < 1) {
        cfg.gridDim = dim3(unsigned(gg.parts), 1, 1);
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, fn, &cfg) != cudaSuccess || nc < 1) {
            cudaGetLastError();
            return SAMPLER_ERR_CUDA;
        }
        h->grp_occ[slot] = nc;
        h->grp_occ_smem[slot] = gg.smem;
    }
    const int clusters = std::max(1, std::min(h->grp_occ[slot], p.n_chunks));
    cfg.gridDim = dim3(unsigned(clusters * gg.parts), 1, 1);
    void* args[] = {&p};
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

int launch(sampler_t h, const sampler_args_t* a, cudaStream_t stream)
{
    ColGeometry cg;
    if (col_eligible(h, a, &cg)) return launch_col(h, a, cg, stream);
    {
        GroupGeometry gg;
        const int es = a->dtype == SAMPLER_DTYPE_BF16 ? 2 : 4;
        if (!(h->flags & SAMPLER_CREATE_ROW_KERNEL) && group_geometry(a->vocab, es, a->hist_offsets != nullptr, &gg))
            return launch_group(h, a, gg, stream);
    }
    const bool pen = a->hist_offsets != nullptr;
    const int esize = a->dtype == SAMPLER_DTYPE_BF16 ? 2 : 4;
    const Geometry g = geometry(a->vocab, esize, pen);
    if (g.smem > size_t(kMaxSmem)) return SAMPLER_ERR_TOO_LARGE;
    void* fn = pick_kernel(a->dtype, pen);
    const int slot = kernel_slot(a->dtype, pen);
    if (h->smem_set[slot] < g.smem) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(g.smem)) !=
            cudaSuccess)
            return SAMPLER_ERR_CUDA;
        h->smem_set[slot] = g.smem;
    }

    dst::KernelParams p;
    std::memset(&p, 0, sizeof p);
    p.logits = a->logits;
    p.vocab = a->vocab;
    p.row_stride = a->row_stride;
    p.n_logit_rows = a->n_logit_rows > 0 ? a->n_logit_rows : a->n_rows;
    p.logit_row = a->logit_row;
    p.temperature = a->temperature;
    p.top_k = a->top_k;
    p.top_p = a->top_p;
    p.min_p = a->min_p;
    p.presence = a->presence_penalty;
    p.frequency = a->frequency_penalty;
    p.repetition = a->repetition_penalty;
    p.seed = a->seed;
    p.has_seed = a->has_seed;
    p.stream_id = a->stream_id;
    p.hist_offsets = a->hist_offsets;
    p.hist_ids = a->hist_ids;
    p.global_seed = a->global_seed;
    p.philox_offset = a->philox_offset;
    p.philox_offset_dev = a->philox_offset_dev;
    p.out_tokens = a->out_tokens;
    p.out_probs = a->out_probs;
    p.out_logprobs = a->out_logprobs;
    p.out_status = a->out_status;
    p.slice_len = g.slice;

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(unsigned(a->n_rows * g.cluster), 1, 1);
    cfg.blockDim = dim3(dst::kThreads, 1, 1);
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(g.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

// Units of one row: about one per warp of the GPU, between kUnitMinElems (or the
// whole row) and one warp's slot; a multiple of 16 bytes.
ColGeometry col_geometry(int64_t N, int64_t V, int esize, int sms)
{
    ColGeometry g;
    const int64_t epv = 16 / esize;
    const int64_t w_min = dst::col::kUnitMinElems;
    const int64_t w_max = dst::col::kSlotBytes / esize;
    const int64_t warps = int64_t(sms) * dst::col::kW;
    const int64_t g0 = std::max<int64_t>(1, warps / std::max<int64_t>(N, 1));
    int64_t w = (V + g0 - 1) / g0;
    w = (w + epv - 1) / epv * epv;
    w = std::min(std::max(w, w_min), w_max);
    w = std::min(w, (V + epv - 1) / epv * epv);
    g.w = int(w);
    g.gc = int((V + w - 1) / w);
    g.units = N * g.gc;
    // enough CTAs for one unit per warp and one per row (rows finish in parallel),
    // at most one per SM (all co-resident)
    const int64_t want = std::max<int64_t>((g.units + dst::col::kW - 1) / dst::col::kW, std::max<int64_t>(N, 1));
    g.grid = int(std::min<int64_t>(sms, want));
    return g;
}

// Largest unit count col_geometry gives for up to `rows` rows of up to `vocab`.
int64_t col_max_units(int64_t rows, int64_t vocab, int sms)
{
    int64_t best = 0;
    for (int esize = 2; esize <= 4; esize += 2)
        for (int64_t n = 1; n <= rows; ++n) best = std::max(best, col_geometry(n, vocab, esize, sms).units);
    return best;
}

// The unit-split kernel serves small batches without penalties or outputs.
bool col_eligible(sampler_t h, const sampler_args_t* a, ColGeometry* g)
{
    if (!h->col_rec || a->n_rows > h->col_rows) return false;
    if (a->hist_offsets || a->out_probs || a->out_logprobs) return false;
    const int esize = a->dtype == SAMPLER_DTYPE_BF16 ? 2 : 4;
    *g = col_geometry(a->n_rows, a->vocab, esize, h->num_sms);
    return g->units <= h->col_units && g->gc <= dst::col::kMaxUnits;
}

template <typename InT>
void* col_kernel() { return reinterpret_cast<void*>(&dst::col::colsplit_kernel<InT>); }

void fill_col_params(dst::col::ColParams& p, const sampler_args_t* a, const ColGeometry& g)
{
    std::memset(&p, 0, sizeof p);
    dst::KernelParams& k = p.k;
    k.logits = a->logits;
    k.vocab = a->vocab;
    k.row_stride = a->row_stride;
    k.n_logit_rows = a->n_logit_rows > 0 ? a->n_logit_rows : a->n_rows;
    k.logit_row = a->logit_row;
    k.temperature = a->temperature;
    k.top_k = a->top_k;
    k.top_p = a->top_p;
    k.min_p = a->min_p;
    k.presence = a->presence_penalty;
    k.frequency = a->frequency_penalty;
    k.repetition = a->repetition_penalty;
    k.seed = a->seed;
    k.has_seed = a->has_seed;
    k.stream_id = a->stream_id;
    k.global_seed = a->global_seed;
    k.philox_offset = a->philox_offset;
    k.philox_offset_dev = a->philox_offset_dev;
    k.out_tokens = a->out_tokens;
    k.out_status = a->out_status;
    p.n_rows = int(a->n_rows);
    p.gc = g.gc;
    p.w = g.w;
    p.n_units = int(g.units);
}

// A cooperative launch: a row's finishing CTA waits for units on other CTAs, so all
// must be resident.
int launch_col_kernel(void* fn, dst::col::ColParams& p, const ColGeometry& g, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(g.grid);
    cfg.blockDim = dim3(dst::col::kT);
    cfg.dynamicSmemBytes = dst::col::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

int launch_col(sampler_t h, const sampler_args_t* a, const ColGeometry& g, cudaStream_t stream)
{
    const bool bf = a->dtype == SAMPLER_DTYPE_BF16;
    void* fn = bf ? col_kernel<uint16_t>() : col_kernel<float>();
    const int slot = bf ? 1 : 0;
    if (h->col_smem_set[slot] < dst::col::kSmemBytes) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dst::col::kSmemBytes)) !=
            cudaSuccess)
            return SAMPLER_ERR_CUDA;
        h->col_smem_set[slot] = dst::col::kSmemBytes;
    }
    dst::col::ColParams p;
    fill_col_params(p, a, g);
    p.rec = h->col_rec;
    p.sync = h->col_bar;
    p.stats = h->stats;
    return launch_col_kernel(fn, p, g, stream);
}

int check_args(sampler_t h, const sampler_args_t* a)
{
    if (!h || !a) return SAMPLER_ERR_NULL_ARG;
    if (a->n_rows < 0 || a->vocab < 1 || a->row_stride < a->vocab || a->n_logit_rows < 0)
        return SAMPLER_ERR_BAD_SHAPE;
    if (a->dtype != SAMPLER_DTYPE_F32 && a->dtype != SAMPLER_DTYPE_BF16) return SAMPLER_ERR_BAD_DTYPE;
    if (a->n_rows > h->max_rows || a->vocab > h->max_vocab) return SAMPLER_ERR_TOO_LARGE;
    if (a->n_rows == 0) return SAMPLER_OK;
    if (!a->logits || !a->temperature || !a->out_tokens) return SAMPLER_ERR_NULL_ARG;
    if (a->has_seed && !a->seed) return SAMPLER_ERR_NULL_ARG;
    if (a->hist_offsets && !a->hist_ids) return SAMPLER_ERR_NULL_ARG;
    return SAMPLER_OK;
}

}  // namespace

// ---------------------------------------------------------------- allocation-free entry
// The unit-split kernel's workspace (the per-row counters, then the per-(row, unit)
// records) lives in this module's own device memory for sampler_sample_noalloc.
namespace {

constexpr int kNoAllocRows = SAMPLER_NOALLOC_MAX_ROWS;
constexpr size_t kNoAllocCounterBytes = 2048;  // the per-row counters, padded
constexpr size_t kNoAllocScratchBytes = size_t(9) << 19;  // 4.5 MiB: 64 rows of up to 262144
constexpr int64_t kNoAllocUnits =
    int64_t((kNoAllocScratchBytes - kNoAllocCounterBytes) / sizeof(dst::col::ColRec));
static_assert(sizeof(dst::col::RowSync) <= kNoAllocCounterBytes, "row counter area");
static_assert(kNoAllocCounterBytes % alignof(dst::col::ColRec) == 0, "record alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
    bool ready;
    int num_sms;
    unsigned char* scratch;  // device address of g_noalloc_scratch on this device
    size_t smem_set[2];
};

std::mutex g_noalloc_mutex;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Once per device (the device current): find the scratch array's address, read
// the SM count and clear the per-row counters, which must start at zero (every
// launch leaves them at zero).
int noalloc_setup(int dev, cudaStream_t stream, NoAllocDevice* out)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice& d = g_noalloc_dev[dev];
    if (!d.ready) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, col_kernel<uint16_t>()) != cudaSuccess) {
            cudaGetLastError();
            return SAMPLER_ERR_NO_DEVICE;
        }
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SAMPLER_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            return SAMPLER_ERR_CUDA;
        if (cudaMemsetAsync(ptr, 0, kNoAllocCounterBytes, stream) != cudaSuccess) return SAMPLER_ERR_CUDA;
        d.scratch = static_cast<unsigned char*>(ptr);
        d.num_sms = sms;
        std::memset(d.smem_set, 0, sizeof d.smem_set);
        d.ready = true;
    }
    *out = d;
    return SAMPLER_OK;
}

int noalloc_grant_smem(int dev, int slot, void* fn, size_t smem)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice& d = g_noalloc_dev[dev];
    if (d.smem_set[slot] < smem) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
            return SAMPLER_ERR_CUDA;
        d.smem_set[slot] = smem;
    }
    return SAMPLER_OK;
}

}  // namespace

extern "C" {

uint32_t sampler_abi_version(void) { return (1u << 16) | 0u; }

int sampler_get_stat(sampler_t h, int which, uint64_t* value, int reset)
{
    if (!h || !value) return SAMPLER_ERR_NULL_ARG;
    if (which < 0 || which >= kNumStats) return SAMPLER_ERR_BAD_SHAPE;
    if (cudaSetDevice(h->device) != cudaSuccess) return SAMPLER_ERR_CUDA;
    unsigned long long v = 0;
    if (cudaMemcpy(&v, h->stats + which, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SAMPLER_ERR_CUDA;
    if (reset && cudaMemset(h->stats + which, 0, sizeof v) != cudaSuccess) return SAMPLER_ERR_CUDA;
    *value = v;
    return SAMPLER_OK;
}

const char* sampler_status_string(int code)
{
    switch (code) {
        case SAMPLER_OK: return "ok";
        case SAMPLER_ERR_NULL_ARG: return "a required pointer is NULL";
        case SAMPLER_ERR_BAD_SHAPE: return "bad shape (rows, vocab or row stride)";
        case SAMPLER_ERR_TOO_LARGE: return "rows or vocab above the handle's limits";
        case SAMPLER_ERR_BAD_DTYPE: return "unknown logits dtype";
        case SAMPLER_ERR_CUDA: return "a CUDA call failed";
        case SAMPLER_ERR_NO_DEVICE: return "no usable sm_103 device";
        case SAMPLER_ERR_NO_STAGING: return "handle has no host staging buffers";
        case SAMPLER_ERR_UNSUPPORTED: return "not supported by this entry point";
        case SAMPLER_ROW_NONFINITE: return "row: NaN or +inf logit";
        case SAMPLER_ROW_ALL_NEG_INF: return "row: every logit is -inf";
        case SAMPLER_ROW_BAD_PARAM: return "row: parameter out of range";
        case SAMPLER_ROW_BAD_HISTORY: return "row: history id out of range or history too long";
        case SAMPLER_ROW_TIMEOUT: return "row: internal wait gave up";
        default: return "unknown code";
    }
}

int sampler_create(sampler_t* out, const sampler_config_t* cfg)
{
    if (!out) return SAMPLER_ERR_NULL_ARG;
    *out = nullptr;
    if (!cfg) return SAMPLER_ERR_NULL_ARG;
    if (cfg->max_rows < 1 || cfg->max_vocab < 1 || cfg->max_vocab > kMaxVocabLimit ||
        cfg->max_history < 0)
        return SAMPLER_ERR_BAD_SHAPE;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || cfg->device < 0 || cfg->device >= ndev)
        return SAMPLER_ERR_NO_DEVICE;
    if (cudaSetDevice(cfg->device) != cudaSuccess) return SAMPLER_ERR_NO_DEVICE;
    // the kernels are built for sm_103a only: make sure the image loads here
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, pick_kernel(SAMPLER_DTYPE_F32, false)) != cudaSuccess) {
        cudaGetLastError();
        return SAMPLER_ERR_NO_DEVICE;
    }
    sampler_s* h = new (std::nothrow) sampler_s;
    if (!h) return SAMPLER_ERR_CUDA;
    std::memset(h, 0, sizeof *h);
    h->device = cfg->device;
    h->max_rows = cfg->max_rows;
    h->max_vocab = cfg->max_vocab;
    h->max_history = cfg->max_history;
    h->flags = cfg->flags;
    cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, cfg->device);
    h->col_rows = int(std::min<int64_t>(cfg->max_rows, dst::col::kMaxRows));
    h->col_units = col_max_units(h->col_rows, cfg->max_vocab, h->num_sms);
    {
        const size_t rec_bytes = size_t(h->col_units) * sizeof(dst::col::ColRec);
        if (cudaMalloc(&h->col_rec, rec_bytes) != cudaSuccess ||
            cudaMalloc(&h->col_bar, sizeof(dst::col::RowSync)) != cudaSuccess ||
            cudaMemset(h->col_bar, 0, sizeof(dst::col::RowSync)) != cudaSuccess ||
            cudaMalloc(&h->stats, kNumStats * sizeof(unsigned long long)) != cudaSuccess ||
            cudaMemset(h->stats, 0, kNumStats * sizeof(unsigned long long)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            cudaFree(h->col_rec);
            cudaFree(h->col_bar);
            cudaFree(h->stats);
            delete h;
            return SAMPLER_ERR_CUDA;
        }
    }
    if (cfg->flags & SAMPLER_CREATE_HOST_STAGING) {
        const size_t R = size_t(cfg->max_rows), V = size_t(cfg->max_vocab);
        size_t bytes = 0;
        bytes += align16(R * V * 4);          // logits (largest element type)
        bytes += 2 * align16(R * V * 4);      // probs, logprobs
        bytes += 16 * align16(R * 8);         // per-row arrays
        bytes += align16((R + 1) * 4) + align16(size_t(cfg->max_history) * 4 + 4);
        if (cudaMalloc(&h->stage_base, bytes) != cudaSuccess) {
            cudaFree(h->col_rec);
            cudaFree(h->col_bar);
            cudaFree(h->stats);
            delete h;
            return SAMPLER_ERR_CUDA;
        }
        h->stage_bytes = bytes;
    }
    *out = h;
    return SAMPLER_OK;
}

void sampler_destroy(sampler_t h)
{
    if (!h) return;
    int cur = -1;
    cudaGetDevice(&cur);
    cudaSetDevice(h->device);
    if (h->stage_base) cudaFree(h->stage_base);
    if (h->col_rec) cudaFree(h->col_rec);
    if (h->col_bar) cudaFree(h->col_bar);
    if (h->stats) cudaFree(h->stats);
    if (cur >= 0) cudaSetDevice(cur);
    delete h;
}

int sampler_sample(sampler_t h, const sampler_args_t* a, sampler_stream_t stream)
{
    int rc = check_args(h, a);
    if (rc != SAMPLER_OK || a->n_rows == 0) return rc;
    if (cudaSetDevice(h->device) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return launch(h, a, reinterpret_cast<cudaStream_t>(stream));
}

int sampler_sample_noalloc(const sampler_args_t* a, sampler_stream_t stream_)
{
    if (!a) return SAMPLER_ERR_NULL_ARG;
    if (a->n_rows < 0 || a->vocab < 1 || a->row_stride < a->vocab || a->n_logit_rows < 0)
        return SAMPLER_ERR_BAD_SHAPE;
    if (a->dtype != SAMPLER_DTYPE_F32 && a->dtype != SAMPLER_DTYPE_BF16) return SAMPLER_ERR_BAD_DTYPE;
    if (a->n_rows > kNoAllocRows || a->vocab > kMaxVocabLimit) return SAMPLER_ERR_TOO_LARGE;
    if (a->hist_offsets || a->hist_ids || a->out_probs || a->out_logprobs) return SAMPLER_ERR_UNSUPPORTED;
    if (a->n_rows == 0) return SAMPLER_OK;
    if (!a->logits || !a->temperature || !a->out_tokens) return SAMPLER_ERR_NULL_ARG;
    if (a->has_seed && !a->seed) return SAMPLER_ERR_NULL_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
        return SAMPLER_ERR_NO_DEVICE;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    NoAllocDevice d;
    int rc = noalloc_setup(dev, stream, &d);
    if (rc != SAMPLER_OK) return rc;
    const bool bf = a->dtype == SAMPLER_DTYPE_BF16;
    const ColGeometry g = col_geometry(a->n_rows, a->vocab, bf ? 2 : 4, d.num_sms);
    if (g.units > kNoAllocUnits || g.gc > dst::col::kMaxUnits) return SAMPLER_ERR_TOO_LARGE;
    void* fn = bf ? col_kernel<uint16_t>() : col_kernel<float>();
    rc = noalloc_grant_smem(dev, bf ? 1 : 0, fn, dst::col::kSmemBytes);
    if (rc != SAMPLER_OK) return rc;
    dst::col::ColParams p;
    fill_col_params(p, a, g);
    p.sync = reinterpret_cast<dst::col::RowSync*>(d.scratch);
    p.rec = reinterpret_cast<dst::col::ColRec*>(d.scratch + kNoAllocCounterBytes);
    p.stats = nullptr;
    return launch_col_kernel(fn, p, g, stream);
}

int sampler_sample_host(sampler_t h, const sampler_args_t* a, sampler_stream_t stream_)
{
    int rc = check_args(h, a);
    if (rc != SAMPLER_OK || a->n_rows == 0) return rc;
    if (!h->stage_base) return SAMPLER_ERR_NO_STAGING;
    const int64_t N = a->n_rows, V = a->vocab;
    const int64_t NL = a->n_logit_rows > 0 ? a->n_logit_rows : N;
    if (NL > h->max_rows) return SAMPLER_ERR_TOO_LARGE;
    int64_t hist_len = 0;
    if (a->hist_offsets) {
        hist_len = a->hist_offsets[N];
        if (hist_len < 0 || hist_len > h->max_history) return SAMPLER_ERR_TOO_LARGE;
    }
    if (cudaSetDevice(h->device) != cudaSuccess) return SAMPLER_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
    const size_t R = size_t(h->max_rows), VM = size_t(h->max_vocab);
    const int esize = a->dtype == SAMPLER_DTYPE_BF16 ? 2 : 4;

    unsigned char* cur = h->stage_base;
    auto take = [&](size_t bytes) {
        unsigned char* p = cur;
        cur += align16(bytes);
        return p;
    };
    unsigned char* d_logits = take(R * VM * 4);
    float* d_probs = reinterpret_cast<float*>(take(R * VM * 4));
    float* d_logprobs = reinterpret_cast<float*>(take(R * VM * 4));
    sampler_args_t d = *a;
    bool fail = false;
    auto put = [&](const void* src, size_t elem) -> void* {
        unsigned char* p = take(R * 8);
        if (src && cudaMemcpyAsync(p, src, size_t(N) * elem, cudaMemcpyHostToDevice, st) != cudaSuccess)
            fail = true;
        return src ? p : nullptr;
    };
    // logits: compact NL rows of V elements
    if (cudaMemcpy2DAsync(d_logits, size_t(V) * esize, a->logits, size_t(a->row_stride) * esize,
                          size_t(V) * esize, size_t(NL), cudaMemcpyHostToDevice, st) != cudaSuccess)
        fail = true;
    d.logits = d_logits;
    d.row_stride = V;
    d.n_logit_rows = NL;
    d.logit_row = static_cast<const int32_t*>(put(a->logit_row, 4));
    d.temperature = static_cast<const float*>(put(a->temperature, 4));
    d.top_k = static_cast<const int32_t*>(put(a->top_k, 4));
    d.top_p = static_cast<const float*>(put(a->top_p, 4));
    d.min_p = static_cast<const float*>(put(a->min_p, 4));
    d.presence_penalty = static_cast<const float*>(put(a->presence_penalty, 4));
    d.frequency_penalty = static_cast<const float*>(put(a->frequency_penalty, 4));
    d.repetition_penalty = static_cast<const float*>(put(a->repetition_penalty, 4));
    d.seed = static_cast<const uint64_t*>(put(a->seed, 8));
    d.has_seed = static_cast<const uint8_t*>(put(a->has_seed, 1));
    d.stream_id = static_cast<const uint32_t*>(put(a->stream_id, 4));
    int32_t* d_tokens = static_cast<int32_t*>(static_cast<void*>(take(R * 8)));
    int32_t* d_status = static_cast<int32_t*>(static_cast<void*>(take(R * 8)));
    d.out_tokens = d_tokens;
    d.out_status = a->out_status ? d_status : nullptr;
    d.out_probs = a->out_probs ? d_probs : nullptr;
    d.out_logprobs = a->out_logprobs ? d_logprobs : nullptr;
    d.philox_offset_dev = nullptr;
    unsigned char* d_hoff = take((R + 1) * 4);
    unsigned char* d_hids = take(size_t(h->max_history) * 4 + 4);
    if (a->hist_offsets) {
        if (cudaMemcpyAsync(d_hoff, a->hist_offsets, size_t(N + 1) * 4, cudaMemcpyHostToDevice, st) !=
            cudaSuccess)
            fail = true;
        if (hist_len > 0 &&
            cudaMemcpyAsync(d_hids, a->hist_ids, size_t(hist_len) * 4, cudaMemcpyHostToDevice, st) !=
                cudaSuccess)
            fail = true;
        d.hist_offsets = reinterpret_cast<const int32_t*>(d_hoff);
        d.hist_ids = reinterpret_cast<const int32_t*>(d_hids);
    }
    if (fail) return SAMPLER_ERR_CUDA;
    rc = launch(h, &d, st);
    if (rc != SAMPLER_OK) return rc;
    if (cudaMemcpyAsync(a->out_tokens, d_tokens, size_t(N) * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SAMPLER_ERR_CUDA;
    if (a->out_status &&
        cudaMemcpyAsync(a->out_status, d_status, size_t(N) * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SAMPLER_ERR_CUDA;
    if (a->out_probs && cudaMemcpyAsync(a->out_probs, d_probs, size_t(N * V) * 4,
                                        cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SAMPLER_ERR_CUDA;
    if (a->out_logprobs && cudaMemcpyAsync(a->out_logprobs, d_logprobs, size_t(N * V) * 4,
                                           cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SAMPLER_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

}  // extern "C"
