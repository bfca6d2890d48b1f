// Partition-kernel instantiations for float caches.
#include "attention_dispatch.cuh"

namespace pkvd {
cudaError_t partition_f32(const PartParams& pp, int D, int hpw, int gmax, int path, int grid, size_t smem,
                         cudaStream_t st) {
  return dispatch_partition<float>(pp, D, hpw, gmax, path, grid, smem, st);
}
}  // namespace pkvd
