// decode_f16.cu -- instantiates the paged decode kernels for __half pools.
#include "decode.cuh"

namespace pkv {

template <>
cudaError_t launch_decode<__half>(const DecodeParams& p, int head_dim, int group, cudaStream_t stream) {
    return launch_decode_impl<__half>(p, head_dim, group, stream);
}

}  // namespace pkv
