// fp16 instantiations of the paged decode kernel.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f16(int head_dim, bool split, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream) {
    if (head_dim == 64) return launch_decode_t<__half, 64>(split, tmk, tmv, p, grid, stream);
    return launch_decode_t<__half, 128>(split, tmk, tmv, p, grid, stream);
}

}  // namespace pa
