// nq_decompress_delta.cu -- the head_dim 96 / 128 decoders of tensors with a
// temporal delta (the kernels of nq_decompress.cuh with DELTA set).
#include "nq_decompress.cuh"

namespace nq {

int launch_wide_delta(const LaunchArgs& a, int d, int bits, bool joint, const uint8_t* idx, const uint16_t* coset,
                      const __half* scales, const float4* rope, const CUtensorMap& map, const ChainState& cs) {
    return launch_wide_as<true>(a, d, bits, joint, idx, coset, scales, rope, map, cs);
}

}  // namespace nq
