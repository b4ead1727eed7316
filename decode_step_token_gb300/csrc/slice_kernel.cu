// slice_kernel.cu -- geometry and launch of the slice kernel (design in
// slice_sampler.cuh), and its variant without the extensions of
// sampler_sample_ex (the others are built in slice_kernel_ext.cu).
#include <algorithm>
#include <cstring>

#include "launch.h"

#define SLC_FILTERS 0
#define SLC_LP 0
#define SLC_VARIANT base
#include "slice_kernel.cuh"
#undef SLC_FILTERS
#undef SLC_LP
#undef SLC_VARIANT

namespace dst {

static_assert(sizeof(slc::SliceHdr) == 16, "slice header layout");
static_assert(sizeof(slc::SliceBody) % 16 == 0, "slice body alignment");
static_assert(slc::kMaxRows <= slc::kT, "one thread per row classifies the batch");
static_assert(slc::kHead < slc::kMaxSmem, "shared-memory head");

static_assert(kSliceMaxRows == slc::kMaxRows && kSliceMaxSlices == slc::kMaxSlices, "slice limits");
static_assert(slc::kMaxTopN == SAMPLER_MAX_TOP_N && slc::kMaxBias == SAMPLER_MAX_BIAS &&
                  slc::kMaxStop == SAMPLER_MAX_STOP, "extension limits");
static_assert(kSliceHdrBytes == sizeof(slc::SliceHdr) && kSliceBodyBytes == sizeof(slc::SliceBody),
              "slice record sizes");
static_assert(kSliceCntStride == slc::kCntStride, "counter stride");

namespace {

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// The kernel for the logits' type and the extensions a call asks for (0: none,
// 1: filters only, 2: logprob outputs, with or without filters).
void* kernel_of(int dtype, int variant)
{
    if (variant) return slice_ext_kernel(dtype, variant == 2);
    return dtype == SAMPLER_DTYPE_BF16 ? reinterpret_cast<void*>(&slc::base::slice_kernel<uint16_t>)
                                       : reinterpret_cast<void*>(&slc::base::slice_kernel<float>);
}

}  // namespace

bool kernels_loadable()
{
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel_of(SAMPLER_DTYPE_F32, 0)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return true;
}

bool slice_geometry(int64_t N, int64_t V, int esize, int sms, SliceGeometry* g)
{
    if (N < 1 || N > slc::kMaxRows || V < 1 || sms < 1) return false;
    const int64_t epv = 16 / esize;
    const int64_t wmax = int64_t(slc::kSlotBytes) / esize / epv * epv;  // one warp's slot
    // about one unit per warp of the GPU, each between kMinUnit elements (or the
    // whole row) and one slot
    const int64_t gs_min = (V + wmax - 1) / wmax;
    const int64_t gs_max = std::max<int64_t>(gs_min, (V + slc::kMinUnit - 1) / slc::kMinUnit);
    const int64_t gs_want = (int64_t(sms) * slc::kW + N - 1) / N;
    int64_t G = std::min(std::max(gs_want, gs_min), gs_max);
    if (G > slc::kMaxSlices) return false;
    const int64_t W = std::min(wmax, round_up((V + G - 1) / G, epv));
    G = (V + W - 1) / W;
    if (G > slc::kMaxSlices) return false;
    const int64_t units = N * G;
    g->G = int(G);
    g->W = int(W);
    g->units = int(units);
    g->ctas = int(std::min<int64_t>(sms, (units + slc::kW - 1) / slc::kW));
    g->smem = slc::kSmemBytes;
    return true;
}

int slice_prepare(int dtype, size_t smem)
{
    for (int variant = 0; variant < 3; ++variant)
        if (cudaFuncSetAttribute(kernel_of(dtype, variant), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

int slice_launch(const sampler_args_t* a, const sampler_ext_t* lp, const SliceGeometry& g,
                 const SliceWorkspace& ws, uint32_t max_polls, bool pdl, cudaStream_t stream)
{
    slc::SliceParams p;
    std::memset(&p, 0, sizeof p);
    KernelParams& k = p.k;
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
    if (lp) {
        k.out_tok_lp = lp->out_token_logprob;
        k.top_n = lp->top_n;
        k.out_top_ids = lp->top_n > 0 ? lp->out_top_ids : nullptr;
        k.out_top_lp = lp->top_n > 0 ? lp->out_top_logprobs : nullptr;
        k.lp_unscaled = lp->unscaled ? 1 : 0;
        k.vocab_mask = lp->vocab_mask;
        k.mask_stride = lp->mask_stride;
        k.bias_offsets = lp->bias_offsets;
        k.bias_ids = lp->bias_ids;
        k.bias_values = lp->bias_values;
        k.min_tokens_left = lp->min_tokens_left;
        k.stop_offsets = lp->stop_offsets;
        k.stop_ids = lp->stop_ids;
        k.sanitize_nan = lp->sanitize_nan ? 1 : 0;
    }
    p.n_rows = int(a->n_rows);
    p.G = g.G;
    p.W = g.W;
    p.n_units = g.units;
    p.hdr = static_cast<slc::SliceHdr*>(ws.hdr);
    p.body = static_cast<slc::SliceBody*>(ws.body);
    p.cnt = ws.cnt;
    p.stats = ws.stats;
    p.max_polls = max_polls;
    p.pdl = pdl ? 1 : 0;

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(unsigned(g.ctas));
    cfg.blockDim = dim3(slc::kT);
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const int variant = !lp ? 0 : (lp->out_token_logprob || lp->top_n > 0) ? 2 : 1;
    void* fn = kernel_of(a->dtype, variant);
    void* args[] = {&p};
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

}  // namespace dst
