// fp16 instantiations of the paged decode kernel.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f16(int head_dim, int mode, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream) {
    if (head_dim == 64) return launch_decode_t<__half, 64>(mode, tmk, tmv, p, grid, stream);
    return launch_decode_t<__half, 128>(mode, tmk, tmv, p, grid, stream);
}

cudaError_t launch_decode_fp8_f16(int mode, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    return launch_decode_fp8_t<__half>(mode, tmk, tmv, p, grid, stream);
}

}  // namespace pa
