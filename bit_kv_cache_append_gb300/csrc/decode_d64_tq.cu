// TurboQuant decode kernels for head_dim 64.
#include "decode_kivi.cuh"

namespace kvq {
template cudaError_t launch_tq_d<64>(DecodeArgs& a, cudaStream_t s, int sm_count);
}  // namespace kvq
