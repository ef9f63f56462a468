// fd_gqa_bf16.cu -- the grouped-query decode kernel instantiated for bf16 K/V.
#include "fd_gqa_kernel.cuh"

namespace fd {

cudaError_t launch_gqa_bf16(int d, const GqaParams &gp, cudaStream_t s)
{
    return launch_gqa_dt<__nv_bfloat16>(d, gp, s);
}

}  // namespace fd
