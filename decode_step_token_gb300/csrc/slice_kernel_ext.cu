// slice_kernel_ext.cu -- the slice kernel's variant with the extensions of
// sampler_sample_ex (logprob outputs, vocabulary mask, logit_bias, min_tokens,
// NaN sanitising); its own translation unit so that the two variants compile
// side by side.
#include "launch.h"

#define SLC_EXT 1
#define SLC_VARIANT ext
#include "slice_kernel.cuh"
#undef SLC_EXT
#undef SLC_VARIANT

namespace dst {

void* slice_ext_kernel(int dtype)
{
    return dtype == SAMPLER_DTYPE_BF16 ? reinterpret_cast<void*>(&slc::ext::slice_kernel<uint16_t>)
                                       : reinterpret_cast<void*>(&slc::ext::slice_kernel<float>);
}

}  // namespace dst
