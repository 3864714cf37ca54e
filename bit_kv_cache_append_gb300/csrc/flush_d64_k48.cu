// KIVI group quantisation (flush.cuh) at head_dim 64, K codes of 4 or 8 bits.
#include "flush.cuh"

namespace kvq {
void launch_flush_d64_k48(const AppendArgs& a, dim3 grid, cudaStream_t s) {
  if (a.geo.kb == 4) launch_flush_kb<64, 4>(a, grid, s);
  else launch_flush_kb<64, 8>(a, grid, s);
}
}  // namespace kvq
