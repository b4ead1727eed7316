// slice_kernel_ext.cu -- the slice kernel's variants with the extensions of
// sampler_sample_ex: the filters alone (vocabulary mask, logit_bias,
// min_tokens, NaN sanitising), and everything (the filters and the logprob
// outputs). A translation unit of their own so that the variants compile side
// by side.
#include "launch.h"

#define SLC_FILTERS 1
#define SLC_LP 0
#define SLC_VARIANT filt
#include "slice_kernel.cuh"
#undef SLC_FILTERS
#undef SLC_LP
#undef SLC_VARIANT

#define SLC_FILTERS 1
#define SLC_LP 1
#define SLC_VARIANT ext
#include "slice_kernel.cuh"
#undef SLC_FILTERS
#undef SLC_LP
#undef SLC_VARIANT

namespace dst {

void* slice_ext_kernel(int dtype, bool lp)
{
    const bool bf = dtype == SAMPLER_DTYPE_BF16;
    if (lp)
        return bf ? reinterpret_cast<void*>(&slc::ext::slice_kernel<uint16_t>)
                  : reinterpret_cast<void*>(&slc::ext::slice_kernel<float>);
    return bf ? reinterpret_cast<void*>(&slc::filt::slice_kernel<uint16_t>)
              : reinterpret_cast<void*>(&slc::filt::slice_kernel<float>);
}

}  // namespace dst
