// Decode kernels instantiated for head_dim 128.
#include "decode_kivi.cuh"

namespace kvq {
cudaError_t launch_kivi_d128(DecodeArgs& a, cudaStream_t s, int sm_count) { return launch_kivi_d<128>(a, s, sm_count); }
}  // namespace kvq
