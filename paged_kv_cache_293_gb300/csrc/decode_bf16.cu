// decode_bf16.cu -- instantiates the paged decode kernels for __nv_bfloat16 pools.
#include "decode.cuh"

namespace pkv {

template <>
cudaError_t launch_decode<__nv_bfloat16>(const DecodeParams& p, int head_dim, int group, cudaStream_t stream) {
    return launch_decode_impl<__nv_bfloat16>(p, head_dim, group, stream);
}

}  // namespace pkv
