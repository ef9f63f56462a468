// fd_gqa_tc.cu -- instantiations of the tcgen05 grouped-query kernel
// (fd_gqa_tc.cuh) for f16 and bf16 K/V at head dims 64 and 128.
#include "fd.h"
#include "fd_gqa_tc.cuh"

namespace fd {

cudaError_t launch_gqa_tc(int dtype, int d, const GqaParams &gp, cudaStream_t s)
{
    if (dtype == FD_BF16)
        return d == 64 ? launch_gqa_tc_t<__nv_bfloat16, 64>(gp, s) : launch_gqa_tc_t<__nv_bfloat16, 128>(gp, s);
    return d == 64 ? launch_gqa_tc_t<__half, 64>(gp, s) : launch_gqa_tc_t<__half, 128>(gp, s);
}

}  // namespace fd
