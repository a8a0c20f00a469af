// decode_f32.cu -- instantiates the paged decode kernels for float pools.
#include "decode.cuh"

namespace pkv {

template <>
cudaError_t launch_decode<float>(const DecodeParams& p, int head_dim, int group, cudaStream_t stream) {
    return launch_decode_impl<float>(p, head_dim, group, stream);
}

}  // namespace pkv
