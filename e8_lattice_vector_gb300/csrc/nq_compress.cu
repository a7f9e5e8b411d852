// nq_compress.cu -- compression launches without a temporal delta, and the
// entry that picks the instantiation (the kernels are in nq_compress.cuh).
#include "nq_compress.cuh"

namespace nq {

int launch_compress_tensor(const LaunchArgs& a, int head_dim, int bits, int mode, const void* x, const float* rope,
                           uint8_t* idx, uint16_t* coset, uint16_t* scales) {
    if (a.delta_chunk > 0) return launch_compress_tensor_delta(a, head_dim, bits, mode, x, rope, idx, coset, scales);
    return launch_compress_tensor_as<false>(a, head_dim, bits, mode, x, rope, idx, coset, scales);
}

}  // namespace nq
