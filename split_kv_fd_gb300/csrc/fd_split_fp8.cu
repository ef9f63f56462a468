// fd_split_fp8.cu -- split-KV decode kernel instantiated for an E4M3 KV cache.
#include "fd_split.cuh"

namespace fd {

cudaError_t launch_split_fp8(int d, const SplitParams &p, size_t smem, cudaStream_t s)
{
    if (d == 64)
        return launch_split_t<__nv_fp8_e4m3, 64>(p, smem, s);
    if (d == 128)
        return launch_split_t<__nv_fp8_e4m3, 128>(p, smem, s);
    if (d == 256)
        return launch_split_t<__nv_fp8_e4m3, 256>(p, smem, s);
    return cudaErrorInvalidValue;
}

}  // namespace fd
