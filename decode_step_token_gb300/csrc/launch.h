// launch.h -- internal interface between the host code of the C ABI
// (sampler_api.cu) and the translation units that hold the kernels. Not part
// of the public header.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "sampler.h"

namespace dst {

struct SliceHdr;   // defined with the slice kernel
struct SliceBody;

// ---------------------------------------------------------------- slice kernel
// Small batches without history and without probs / logprobs outputs.
struct SliceGeometry {
    int G;           // slices per row
    int W;           // elements per slice
    int units;       // rows x slices, one warp's work each
    int ctas;        // grid
    size_t smem;     // dynamic shared memory per CTA
};

struct SliceWorkspace {
    void* hdr;       // [rows][G] 16-byte slice headers
    void* body;      // [rows][G] slice bodies
    uint32_t* cnt;   // [rows * kSliceCntStride] per row: its arrival counter (alone in a 128-byte line)
                     // and a 256-bin histogram of its truncated units' sketch keys; zero between launches
    unsigned long long* stats;  // may be NULL
};

// Limits and record sizes of the slice kernel (checked against its own
// definitions in slice_kernel.cu).
constexpr int kSliceMaxRows = 256;
constexpr int kSliceMaxSlices = 128;
constexpr size_t kSliceHdrBytes = 16;
constexpr size_t kSliceBodyBytes = 464;
constexpr int kSliceCntStride = 32 + 256;  // 32-bit words between two rows' counters (counter line + histogram)

// True when this library's kernels load on the current device.
bool kernels_loadable();

// Geometry for n_rows x vocab of esize-byte logits on `sms` SMs; false when the
// slice kernel does not take the shape.
bool slice_geometry(int64_t n_rows, int64_t vocab, int esize, int sms, SliceGeometry* g);

// Grant the kernel (every variant) its dynamic shared memory (once per device
// and size).
int slice_prepare(int dtype, size_t smem);

// The slice kernel's variants with the extensions of sampler_sample_ex, for the
// logits' type: the filters alone, or (lp) everything (built in
// slice_kernel_ext.cu).
void* slice_ext_kernel(int dtype, bool lp);

// Enqueue one slice-kernel launch. max_polls bounds each wait on a staging copy.
// ext: the step's extensions (NULL: none). pdl: launched as the programmatic
// dependent of the kernel before it on the stream (it waits for that grid
// before it reads the logits).
int slice_launch(const sampler_args_t* a, const sampler_ext_t* ext, const SliceGeometry& g,
                 const SliceWorkspace& ws, uint32_t max_polls, bool pdl, cudaStream_t stream);

// ---------------------------------------------------------------- LM-head GEMM
constexpr int kLmHeadMaxRows = 256;  // hidden rows of one launch (the MMA's N)

struct LmHeadPlan {
    int NT;              // rows rounded up to 16
    int stages;          // operand stages in shared memory
    uint32_t tmem_cols;  // tensor-memory columns (two accumulators)
    int tiles;           // 128-row weight tiles
    int kchunks;         // 64-wide K stages per tile
    int ctas;            // persistent grid
    size_t smem;
};

bool lm_head_plan(int64_t rows, int64_t vocab, int64_t hidden_dim, int sms, LmHeadPlan* plan);
int lm_head_prepare(size_t smem);
// logits [rows, ldl] bf16 = hidden x weight^T; timeouts counts CTAs whose wait gave up.
int lm_head_launch(const sampler_lm_head_t* g, void* logits, int64_t ldl, int64_t rows, int64_t vocab,
                   const LmHeadPlan& plan, unsigned long long* timeouts, cudaStream_t stream);

// ---------------------------------------------------------------- fork-group kernel
// Everything the slice kernel does not take.
struct GroupGeometry {
    int parts;       // CTAs per cluster
    int slice;       // elements per CTA
    int list_cap, part_cap;
    uint32_t off_list, off_cand, off_cnt, off_stage;
    size_t smem;
};

bool group_geometry(int64_t V, int esize, bool pen, GroupGeometry* g);

// Clusters of the fork-group kernel that fit on the device at once (for the
// given variant and shared memory); 0 on error.
int group_occupancy(int dtype, bool pen, const GroupGeometry& g);

int group_prepare(int dtype, bool pen, size_t smem);

// work: two zeroed counters of the handle (the kernel leaves them zeroed)
int group_launch(const sampler_args_t* a, const GroupGeometry& g, int clusters, uint32_t* work, cudaStream_t stream);

}  // namespace dst
