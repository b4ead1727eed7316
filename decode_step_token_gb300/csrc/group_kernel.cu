// group_kernel.cu -- instantiation, geometry and launch of the fork-group kernel
// (design in group_sampler.cuh).
#include <algorithm>
#include <cstring>

#include "group_sampler_kernel.cuh"
#include "launch.h"

namespace dst {

namespace {

constexpr size_t kMaxSmem = 227 * 1024;
constexpr size_t kTwoPerSm = 113 * 1024;  // dynamic shared memory that lets two CTAs share an SM

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

template <typename InT, bool kPen>
void* kernel_ptr()
{
    return reinterpret_cast<void*>(&grp::group_kernel<InT, kPen>);
}

void* kernel_of(int dtype, bool pen)
{
    if (dtype == SAMPLER_DTYPE_BF16) return pen ? kernel_ptr<uint16_t, true>() : kernel_ptr<uint16_t, false>();
    return pen ? kernel_ptr<float, true>() : kernel_ptr<float, false>();
}

}  // namespace

// Parts of at most 64 KB each (up to eight), then the largest candidate lists that
// keep two CTAs per SM; fp32 rows with penalties reuse the count table's space for
// the lists (the counts are folded into the staged row before any list exists).
bool group_geometry(int64_t V, int esize, bool pen, GroupGeometry* g)
{
    const int64_t parts = std::min<int64_t>(grp::kMaxParts, std::max<int64_t>(1, (V * esize + 65535) / 65536));
    int64_t l = (V + parts - 1) / parts;
    l = (l + 15) & ~int64_t(15);
    g->parts = int(parts);
    g->slice = int(l);
    const size_t head = (sizeof(grp::GShared) + 127) & ~size_t(127);
    const size_t stage = align16(size_t(l) * esize + 32);
    const size_t cnt = pen ? align16(size_t(l) * 2 + 16) : 0;
    for (int pass = 0; pass < 2; ++pass) {
        const size_t limit = pass == 0 ? kTwoPerSm : kMaxSmem - 1024;
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

int group_prepare(int dtype, bool pen, size_t smem)
{
    if (cudaFuncSetAttribute(kernel_of(dtype, pen), cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess)
        return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

namespace {

void config_of(const GroupGeometry& g, cudaStream_t stream, cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr)
{
    std::memset(&cfg, 0, sizeof cfg);
    cfg.blockDim = dim3(grp::kT, 1, 1);
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(g.parts);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
}

}  // namespace

int group_occupancy(int dtype, bool pen, const GroupGeometry& g)
{
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    config_of(g, nullptr, cfg, attr);
    cfg.gridDim = dim3(unsigned(g.parts), 1, 1);
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, kernel_of(dtype, pen), &cfg) != cudaSuccess || nc < 1) {
        cudaGetLastError();
        return 0;
    }
    return nc;
}

int group_launch(const sampler_args_t* a, const GroupGeometry& gg, int clusters, uint32_t* work, cudaStream_t stream)
{
    const bool pen = a->hist_offsets != nullptr;
    grp::GroupParams p;
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
    p.chunk = p.group ? grp::kMaxForks : 1;
    p.n_chunks = int((a->n_rows + p.chunk - 1) / p.chunk);
    p.slice_len = gg.slice;
    p.list_cap = gg.list_cap;
    p.part_cap = gg.part_cap;
    p.off_list = gg.off_list;
    p.off_cand = gg.off_cand;
    p.off_cnt = gg.off_cnt;
    p.off_stage = gg.off_stage;
    p.work = work;

    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    config_of(gg, stream, cfg, attr);
    // a persistent grid: as many clusters as fit at once, never more than chunks
    const int nc = std::max(1, std::min(clusters, p.n_chunks));
    cfg.gridDim = dim3(unsigned(nc * gg.parts), 1, 1);
    void* args[] = {&p};
    if (cudaLaunchKernelExC(&cfg, kernel_of(a->dtype, pen), args) != cudaSuccess) return SAMPLER_ERR_CUDA;
    return SAMPLER_OK;
}

}  // namespace dst
