// fd_gqa_f16.cu -- the grouped-query decode kernel instantiated for f16 K/V,
// and the dispatch over storage types.
#include "fd_gqa_kernel.cuh"

namespace fd {

cudaError_t launch_gqa(int dtype, int d, const GqaParams &gp, cudaStream_t s)
{
    return dtype == 2 ? launch_gqa_bf16(d, gp, s) : launch_gqa_dt<__half>(d, gp, s);
}

}  // namespace fd
