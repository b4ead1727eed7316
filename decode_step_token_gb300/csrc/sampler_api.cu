// sampler_api.cu -- the C ABI of libsampler.so (declared in include/sampler.h):
// argument checks, the choice of kernel, the handle's workspace, the
// allocation-free entry point, the host-buffer entry that stages through the
// handle's device buffers, and the LM-head entry. The kernels live in
// slice_kernel.cu, group_kernel.cu and lm_head_kernel.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "launch.h"
#include "sampler.h"

namespace {

constexpr int64_t kMaxVocabLimit = 262144;  // a row always fits one cluster's shared memory
constexpr int kNumStats = 4;
constexpr uint32_t kMaxPolls = 1u << 24;  // bound of each wait on a staging copy

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

int kernel_slot(int dtype, bool pen) { return (dtype == SAMPLER_DTYPE_BF16 ? 2 : 0) + (pen ? 1 : 0); }

// Restores the calling thread's current device when it goes out of scope.
struct DeviceGuard {
    int prev = -1;
    DeviceGuard() { cudaGetDevice(&prev); }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

}  // namespace

struct sampler_s {
    int device;
    int num_sms;
    int64_t max_rows, max_vocab, max_history;
    uint32_t flags;
    uint32_t max_polls;
    // slice kernel: per-(row, slice) records and per-row arrival counters
    dst::SliceWorkspace slice_ws;
    int slice_rows;
    size_t slice_smem_set[2];  // dynamic shared memory already granted per dtype
    // fork-group kernel
    size_t grp_smem_set[4];
    size_t lmh_smem_set;     // LM-head GEMM
    size_t grp_occ_smem[4];  // shared memory of the cached cluster occupancy below
    int grp_occ[4];          // co-resident clusters of the fork-group kernel
    uint32_t* grp_work;      // the fork-group kernel's chunk counters (zero between launches)
    unsigned long long* stats;  // device counters (diagnostics)
    // staging for sampler_sample_host
    unsigned char* stage_base;
    size_t stage_bytes;
};

namespace {

int esize_of(int dtype) { return dtype == SAMPLER_DTYPE_BF16 ? 2 : 4; }

bool slice_takes(const sampler_args_t* a)
{
    return !a->hist_offsets && !a->out_probs && !a->out_logprobs;
}

int launch_group(sampler_t h, const sampler_args_t* a, cudaStream_t stream)
{
    const bool pen = a->hist_offsets != nullptr;
    dst::GroupGeometry gg;
    if (!dst::group_geometry(a->vocab, esize_of(a->dtype), pen, &gg)) return SAMPLER_ERR_TOO_LARGE;
    const int slot = kernel_slot(a->dtype, pen);
    if (h->grp_smem_set[slot] < gg.smem) {
        if (dst::group_prepare(a->dtype, pen, gg.smem) != SAMPLER_OK) return SAMPLER_ERR_CUDA;
        h->grp_smem_set[slot] = gg.smem;
    }
    if (h->grp_occ_smem[slot] != gg.smem || h->grp_occ[slot] < 1) {
        const int nc = dst::group_occupancy(a->dtype, pen, gg);
        if (nc < 1) return SAMPLER_ERR_CUDA;
        h->grp_occ[slot] = nc;
        h->grp_occ_smem[slot] = gg.smem;
    }
    return dst::group_launch(a, gg, h->grp_occ[slot], h->grp_work, stream);
}

// lp: the step's extensions, offered on the slice kernel only (the caller has
// checked that the call takes it). pdl: a slice-kernel launch is the
// programmatic dependent of the kernel enqueued before it.
int launch(sampler_t h, const sampler_args_t* a, cudaStream_t stream, const sampler_ext_t* lp = nullptr,
           bool pdl = false)
{
    dst::SliceGeometry g;
    if (slice_takes(a) && a->n_rows <= h->slice_rows &&
        dst::slice_geometry(a->n_rows, a->vocab, esize_of(a->dtype), h->num_sms, &g)) {
        const int slot = a->dtype == SAMPLER_DTYPE_BF16 ? 1 : 0;
        if (h->slice_smem_set[slot] < g.smem) {
            if (dst::slice_prepare(a->dtype, g.smem) != SAMPLER_OK) return SAMPLER_ERR_CUDA;
            h->slice_smem_set[slot] = g.smem;
        }
        return dst::slice_launch(a, lp, g, h->slice_ws, h->max_polls, pdl, stream);
    }
    if (lp) return SAMPLER_ERR_UNSUPPORTED;
    return launch_group(h, a, stream);
}

// Whether a call with extensions takes the slice kernel (host-visible facts).
bool slice_would_take(sampler_t h, const sampler_args_t* a)
{
    dst::SliceGeometry g;
    return slice_takes(a) && a->n_rows <= h->slice_rows &&
           dst::slice_geometry(a->n_rows, a->vocab, esize_of(a->dtype), h->num_sms, &g);
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

void free_handle(sampler_s* h)
{
    cudaFree(h->slice_ws.hdr);
    cudaFree(h->slice_ws.body);
    cudaFree(h->slice_ws.cnt);
    cudaFree(h->stats);
    cudaFree(h->grp_work);
    cudaFree(h->stage_base);
    delete h;
}

}  // namespace

// ---------------------------------------------------------------- allocation-free entry
// The slice kernel's workspace (the per-row arrival counters, then the per-(row,
// slice) headers and bodies) lives in this module's own device memory for
// sampler_sample_noalloc.
namespace {

constexpr int kNoAllocRows = SAMPLER_NOALLOC_MAX_ROWS;
constexpr size_t kNoAllocCounterBytes = size_t(kNoAllocRows) * dst::kSliceCntStride * sizeof(uint32_t);
constexpr size_t kNoAllocHdrBytes = size_t(kNoAllocRows) * dst::kSliceMaxSlices * dst::kSliceHdrBytes;
constexpr size_t kNoAllocBodyBytes = size_t(kNoAllocRows) * dst::kSliceMaxSlices * dst::kSliceBodyBytes;
constexpr size_t kNoAllocScratchBytes = kNoAllocCounterBytes + kNoAllocHdrBytes + kNoAllocBodyBytes;
static_assert(kNoAllocRows <= dst::kSliceMaxRows, "the slice kernel takes every allowed row count");
static_assert(kNoAllocCounterBytes % 16 == 0 && kNoAllocHdrBytes % 16 == 0, "record alignment");

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
        if (!dst::kernels_loadable()) return SAMPLER_ERR_NO_DEVICE;
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

int noalloc_grant_smem(int dev, int dtype, size_t smem)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice& d = g_noalloc_dev[dev];
    const int slot = dtype == SAMPLER_DTYPE_BF16 ? 1 : 0;
    if (d.smem_set[slot] < smem) {
        if (dst::slice_prepare(dtype, smem) != SAMPLER_OK) return SAMPLER_ERR_CUDA;
        d.smem_set[slot] = smem;
    }
    return SAMPLER_OK;
}

}  // namespace

extern "C" {

uint32_t sampler_abi_version(void) { return (1u << 16) | 3u; }

int sampler_get_stat(sampler_t h, int which, uint64_t* value, int reset)
{
    if (!h || !value) return SAMPLER_ERR_NULL_ARG;
    if (which < 0 || which >= kNumStats) return SAMPLER_ERR_BAD_SHAPE;
    DeviceGuard guard;
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
    DeviceGuard guard;
    if (cudaSetDevice(cfg->device) != cudaSuccess) return SAMPLER_ERR_NO_DEVICE;
    // the kernels are built for sm_103a only: make sure the image loads here
    if (!dst::kernels_loadable()) return SAMPLER_ERR_NO_DEVICE;
    sampler_s* h = new (std::nothrow) sampler_s;
    if (!h) return SAMPLER_ERR_CUDA;
    std::memset(h, 0, sizeof *h);
    h->device = cfg->device;
    h->max_rows = cfg->max_rows;
    h->max_vocab = cfg->max_vocab;
    h->max_history = cfg->max_history;
    h->flags = cfg->flags;
    h->max_polls = (cfg->flags & SAMPLER_CREATE_SHORT_WAITS) ? 0u : kMaxPolls;
    cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, cfg->device);
    h->slice_rows = int(std::min<int64_t>(cfg->max_rows, dst::kSliceMaxRows));
    {
        const size_t recs = size_t(h->slice_rows) * dst::kSliceMaxSlices;
        const size_t cnt_bytes = size_t(h->slice_rows) * dst::kSliceCntStride * sizeof(uint32_t);
        if (cudaMalloc(&h->slice_ws.hdr, recs * dst::kSliceHdrBytes) != cudaSuccess ||
            cudaMalloc(&h->slice_ws.body, recs * dst::kSliceBodyBytes) != cudaSuccess ||
            cudaMalloc(&h->slice_ws.cnt, cnt_bytes) != cudaSuccess ||
            cudaMemset(h->slice_ws.cnt, 0, cnt_bytes) != cudaSuccess ||
            cudaMalloc(&h->stats, kNumStats * sizeof(unsigned long long)) != cudaSuccess ||
            cudaMemset(h->stats, 0, kNumStats * sizeof(unsigned long long)) != cudaSuccess ||
            cudaMalloc(&h->grp_work, 2 * sizeof(uint32_t)) != cudaSuccess ||
            cudaMemset(h->grp_work, 0, 2 * sizeof(uint32_t)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            free_handle(h);
            return SAMPLER_ERR_CUDA;
        }
        h->slice_ws.stats = h->stats;
    }
    if (cfg->flags & SAMPLER_CREATE_HOST_STAGING) {
        const size_t R = size_t(cfg->max_rows), V = size_t(cfg->max_vocab);
        size_t bytes = 0;
        bytes += align16(R * V * 4);          // logits (largest element type)
        bytes += 2 * align16(R * V * 4);      // probs, logprobs
        bytes += 16 * align16(R * 8);         // per-row arrays
        bytes += align16((R + 1) * 4) + align16(size_t(cfg->max_history) * 4 + 4);
        if (cudaMalloc(&h->stage_base, bytes) != cudaSuccess) {
            free_handle(h);
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
    DeviceGuard guard;
    cudaSetDevice(h->device);
    free_handle(h);
}

int sampler_sample(sampler_t h, const sampler_args_t* a, sampler_stream_t stream)
{
    int rc = check_args(h, a);
    if (rc != SAMPLER_OK || a->n_rows == 0) return rc;
    DeviceGuard guard;
    if (cudaSetDevice(h->device) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return launch(h, a, reinterpret_cast<cudaStream_t>(stream));
}

namespace {

// Host checks of a step's extensions; *use is NULL when nothing is asked.
int check_ext(const sampler_args_t* a, const sampler_ext_t* ext, const sampler_ext_t** use)
{
    *use = nullptr;
    if (!ext) return SAMPLER_OK;
    if (ext->top_n < 0 || ext->top_n > SAMPLER_MAX_TOP_N) return SAMPLER_ERR_UNSUPPORTED;
    if (ext->top_n > 0 && (!ext->out_top_ids || !ext->out_top_logprobs)) return SAMPLER_ERR_NULL_ARG;
    if (ext->vocab_mask && ext->mask_stride < (a->vocab + 31) / 32) return SAMPLER_ERR_UNSUPPORTED;
    if (ext->bias_offsets && (!ext->bias_ids || !ext->bias_values)) return SAMPLER_ERR_NULL_ARG;
    if (ext->stop_offsets && !ext->stop_ids) return SAMPLER_ERR_NULL_ARG;
    if (ext->out_token_logprob || ext->top_n > 0 || ext->vocab_mask || ext->bias_offsets || ext->stop_offsets ||
        ext->sanitize_nan)
        *use = ext;
    return SAMPLER_OK;
}

}  // namespace

int sampler_sample_ex(sampler_t h, const sampler_args_t* a, const sampler_ext_t* ext_in, sampler_stream_t stream)
{
    int rc = check_args(h, a);
    if (rc != SAMPLER_OK) return rc;
    const sampler_ext_t* ext = nullptr;
    rc = check_ext(a, ext_in, &ext);
    if (rc != SAMPLER_OK) return rc;
    if (a->n_rows == 0) return SAMPLER_OK;
    DeviceGuard guard;
    if (cudaSetDevice(h->device) != cudaSuccess) return SAMPLER_ERR_CUDA;
    if (ext && !slice_would_take(h, a)) return SAMPLER_ERR_UNSUPPORTED;
    return launch(h, a, reinterpret_cast<cudaStream_t>(stream), ext);
}

namespace {

int check_lm(const sampler_lm_head_t* lm)
{
    if (!lm || !lm->hidden || !lm->weight) return SAMPLER_ERR_NULL_ARG;
    if (lm->hidden_dim < 1 || lm->hidden_stride < lm->hidden_dim || lm->weight_stride < lm->hidden_dim ||
        lm->hidden_stride % 8 != 0 || lm->weight_stride % 8 != 0 ||
        reinterpret_cast<uintptr_t>(lm->hidden) % 16 != 0 || reinterpret_cast<uintptr_t>(lm->weight) % 16 != 0)
        return SAMPLER_ERR_BAD_SHAPE;
    return SAMPLER_OK;
}

// Enqueue the LM-head GEMM (the caller has checked lm and set the device).
int launch_lm_head(sampler_t h, const sampler_lm_head_t* lm, void* logits, int64_t ldl, int64_t rows, int64_t vocab,
                   cudaStream_t stream)
{
    dst::LmHeadPlan plan;
    if (!dst::lm_head_plan(rows, vocab, lm->hidden_dim, h->num_sms, &plan)) return SAMPLER_ERR_TOO_LARGE;
    if (h->lmh_smem_set < plan.smem) {
        if (dst::lm_head_prepare(plan.smem) != SAMPLER_OK) return SAMPLER_ERR_CUDA;
        h->lmh_smem_set = plan.smem;
    }
    return dst::lm_head_launch(lm, logits, ldl, rows, vocab, plan, h->stats + SAMPLER_STAT_LM_HEAD_TIMEOUTS, stream);
}

}  // namespace

int sampler_lm_head(sampler_t h, const sampler_lm_head_t* lm, void* logits, int64_t ldl, int64_t rows,
                    int64_t vocab, sampler_stream_t stream)
{
    if (!h || !logits) return SAMPLER_ERR_NULL_ARG;
    int rc = check_lm(lm);
    if (rc != SAMPLER_OK) return rc;
    if (rows < 1 || vocab < 1 || ldl < vocab) return SAMPLER_ERR_BAD_SHAPE;
    if (rows > SAMPLER_LM_HEAD_MAX_ROWS || vocab > h->max_vocab) return SAMPLER_ERR_TOO_LARGE;
    DeviceGuard guard;
    if (cudaSetDevice(h->device) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return launch_lm_head(h, lm, logits, ldl, rows, vocab, reinterpret_cast<cudaStream_t>(stream));
}

int sampler_lm_head_sample(sampler_t h, const sampler_lm_head_t* lm, const sampler_args_t* a,
                           const sampler_ext_t* ext_in, sampler_stream_t stream_)
{
    int rc = check_args(h, a);
    if (rc != SAMPLER_OK) return rc;
    if (!lm) return SAMPLER_ERR_NULL_ARG;
    const sampler_ext_t* ext = nullptr;
    rc = check_ext(a, ext_in, &ext);
    if (rc != SAMPLER_OK) return rc;
    if (a->n_rows == 0) return SAMPLER_OK;
    if (a->dtype != SAMPLER_DTYPE_BF16) return SAMPLER_ERR_BAD_DTYPE;
    rc = check_lm(lm);
    if (rc != SAMPLER_OK) return rc;
    const int64_t rows = a->n_logit_rows > 0 ? a->n_logit_rows : a->n_rows;
    if (rows > SAMPLER_LM_HEAD_MAX_ROWS) return SAMPLER_ERR_TOO_LARGE;
    DeviceGuard guard;
    if (cudaSetDevice(h->device) != cudaSuccess) return SAMPLER_ERR_CUDA;
    if (ext && !slice_would_take(h, a)) return SAMPLER_ERR_UNSUPPORTED;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    rc = launch_lm_head(h, lm, const_cast<void*>(a->logits), a->row_stride, rows, a->vocab, stream);
    if (rc != SAMPLER_OK) return rc;
    return launch(h, a, stream, ext, true);
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
    dst::SliceGeometry g;
    if (!dst::slice_geometry(a->n_rows, a->vocab, esize_of(a->dtype), d.num_sms, &g)) return SAMPLER_ERR_TOO_LARGE;
    rc = noalloc_grant_smem(dev, a->dtype, g.smem);
    if (rc != SAMPLER_OK) return rc;
    dst::SliceWorkspace ws;
    ws.cnt = reinterpret_cast<uint32_t*>(d.scratch);
    ws.hdr = d.scratch + kNoAllocCounterBytes;
    ws.body = d.scratch + kNoAllocCounterBytes + kNoAllocHdrBytes;
    ws.stats = nullptr;
    return dst::slice_launch(a, nullptr, g, ws, kMaxPolls, false, stream);
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
    DeviceGuard guard;
    if (cudaSetDevice(h->device) != cudaSuccess) return SAMPLER_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
    const size_t R = size_t(h->max_rows), VM = size_t(h->max_vocab);
    const int esize = esize_of(a->dtype);

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
