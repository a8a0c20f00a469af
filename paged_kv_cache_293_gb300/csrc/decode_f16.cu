// decode_f16.cu -- instantiates the paged decode kernels for __half pools: the
// CUDA-core kernel (decode.cuh) and the tensor-core kernel for grouped-query
// heads (decode_mma.cuh), chosen by the engine setting.
#include "decode.cuh"
#include "decode_mma.cuh"
#include "prefix.cuh"

namespace pkv {

template <>
cudaError_t launch_decode<__half>(const DecodeParams& p, int head_dim, int group, cudaStream_t stream) {
    if (use_tensor_cores(group)) {
        const cudaError_t e = launch_decode_mma_impl<__half>(p, head_dim, group, stream);
        if (e != cudaErrorNotSupported) return e;   // else: pool too large for a tensor map
    }
    return launch_decode_impl<__half>(p, head_dim, group, stream);
}

template <>
cudaError_t launch_decode_mma<__half>(const DecodeParams& p, int head_dim, int group,
                                  cudaStream_t stream) {
    return launch_decode_mma_impl<__half>(p, head_dim, group, stream);
}

template <>
cudaError_t launch_prefix<__half>(const PrefixParams& p, const void* k_pool, const void* v_pool,
                               int head_dim, cudaStream_t stream) {
    return launch_prefix_impl<__half>(p, k_pool, v_pool, head_dim, stream);
}

}  // namespace pkv
