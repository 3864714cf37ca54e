// KIVI group quantisation (flush.cuh) at head_dim 128, K codes of 4 or 8 bits.
#include "flush.cuh"

namespace kvq {
void launch_flush_d128_k48(const AppendArgs& a, dim3 grid, cudaStream_t s) {
  if (a.geo.kb == 4) launch_flush_kb<128, 4>(a, grid, s);
  else launch_flush_kb<128, 8>(a, grid, s);
}
}  // namespace kvq
