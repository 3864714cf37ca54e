// KIVI group quantisation (flush.cuh) at head_dim 128, K codes of 2 or 3 bits.
#include "flush.cuh"

namespace kvq {
void launch_flush_d128_k23(const AppendArgs& a, dim3 grid, cudaStream_t s) {
  if (a.geo.kb == 2) launch_flush_kb<128, 2>(a, grid, s);
  else launch_flush_kb<128, 3>(a, grid, s);
}
}  // namespace kvq
