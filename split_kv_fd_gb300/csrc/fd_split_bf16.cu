// fd_split_bf16.cu -- split-KV decode kernel instantiated for bf16 storage.
#include "fd_split.cuh"

namespace fd {

cudaError_t launch_split_bf16(int d, const SplitParams &p, size_t smem, cudaStream_t s)
{
    if (d == 64)
        return launch_split_t<__nv_bfloat16, 64>(p, smem, s);
    if (d == 128)
        return launch_split_t<__nv_bfloat16, 128>(p, smem, s);
    if (d == 256)
        return launch_split_t<__nv_bfloat16, 256>(p, smem, s);
    return cudaErrorInvalidValue;
}

}  // namespace fd
