// nq_compress_delta.cu -- compression launches with a temporal delta (the
// kernels are in nq_compress.cuh).
#include "nq_compress.cuh"

namespace nq {

int launch_compress_tensor_delta(const LaunchArgs& a, int head_dim, int bits, int mode, const void* x,
                                 const float* rope, uint8_t* idx, uint16_t* coset, uint16_t* scales) {
    return launch_compress_tensor_as<true>(a, head_dim, bits, mode, x, rope, idx, coset, scales);
}

}  // namespace nq
