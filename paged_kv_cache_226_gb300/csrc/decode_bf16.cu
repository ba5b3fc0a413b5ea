// bf16 instantiations of the paged decode kernel.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_bf16(int head_dim, int mode, const CUtensorMap& tmk,
                               const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                               cudaStream_t stream) {
    if (head_dim == 64) return launch_decode_t<__nv_bfloat16, 64>(mode, tmk, tmv, p, grid, stream);
    return launch_decode_t<__nv_bfloat16, 128>(mode, tmk, tmv, p, grid, stream);
}

cudaError_t launch_decode_fp8_bf16(int mode, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    return launch_decode_fp8_t<__nv_bfloat16>(mode, tmk, tmv, p, grid, stream);
}

}  // namespace pa
