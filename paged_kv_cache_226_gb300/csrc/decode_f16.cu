// fp16 instantiations of the paged decode kernel.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f16(int head_dim, int mode, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream) {
    if (head_dim == 64) return launch_decode_t<__half, 64>(mode, tmk, tmv, p, grid, stream);
    return launch_decode_t<__half, 128>(mode, tmk, tmv, p, grid, stream);
}

int decode_merge_floats(int head_dim) {
    return head_dim == 64 ? kConsumerWarps * DecodeLayout<64>::kMergeFloatsPerWarp
                          : kConsumerWarps * DecodeLayout<128>::kMergeFloatsPerWarp;
}

cudaError_t launch_decode_fp8_f16(int mode, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    return launch_decode_fp8_t<__half>(mode, tmk, tmv, p, grid, stream);
}

}  // namespace pa
