// KIVI decode kernels for head_dim 64, 8-bit K codes.
#include "decode_kivi.cuh"

namespace kvq {
template cudaError_t launch_kivi_k<64, 8>(DecodeArgs& a, cudaStream_t s, int sm_count);
}  // namespace kvq
