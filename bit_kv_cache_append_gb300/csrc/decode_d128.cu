// Decode kernels instantiated for head_dim 128.
#include "decode_kivi.cuh"

namespace kvq {
cudaError_t launch_kivi_d128(const DecodeArgs& a, cudaStream_t s) { return launch_kivi_d<128>(a, s); }
}  // namespace kvq
