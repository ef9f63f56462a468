// fd_gqa_tc8.cu -- the FP8 tcgen05 grouped-query kernel (fd_gqa_tc8.cuh)
// instantiated for E4M3 K/V at head dim 128.
#include "fd_gqa_tc8.cuh"

namespace fd {

cudaError_t launch_gqa_tc8(int d, const GqaParams &gp, cudaStream_t s)
{
    if (d != 128)
        return cudaErrorInvalidValue;
    return launch_gqa_tc8_t<128>(gp, s);
}

}  // namespace fd
