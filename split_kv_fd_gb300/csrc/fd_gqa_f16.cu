// fd_gqa_f16.cu -- the grouped-query decode kernel instantiated for f16 K/V
// and for E4M3 K/V (converted to f16 in shared memory), and the dispatch over
// storage types.
#include "fd_gqa_kernel.cuh"

namespace fd {

cudaError_t launch_gqa_f8(int d, const GqaParams &gp, cudaStream_t s)
{
    // slices of at most 8 query heads: one column tile
    if (d == 64)
        return gp.pages16 ? launch_gqa_p<__half, 64, 1, true, true>(gp, s)
                          : launch_gqa_p<__half, 64, 1, false, true>(gp, s);
    if (d == 256)
        return gp.pages16 ? launch_gqa_p<__half, 256, 1, true, true>(gp, s)
                          : launch_gqa_p<__half, 256, 1, false, true>(gp, s);
    return gp.pages16 ? launch_gqa_p<__half, 128, 1, true, true>(gp, s)
                      : launch_gqa_p<__half, 128, 1, false, true>(gp, s);
}

cudaError_t launch_gqa(int dtype, int d, const GqaParams &gp, cudaStream_t s)
{
    return dtype == 2 ? launch_gqa_bf16(d, gp, s) : launch_gqa_dt<__half>(d, gp, s);
}

}  // namespace fd
