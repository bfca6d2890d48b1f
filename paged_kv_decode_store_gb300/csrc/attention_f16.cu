// Partition-kernel instantiations for __half caches.
#include "attention_dispatch.cuh"

namespace pkvd {
cudaError_t partition_f16(const PartParams& pp, int D, int hpw, int gmax, int path, int grid, size_t smem,
                         cudaStream_t st) {
  return dispatch_partition<__half>(pp, D, hpw, gmax, path, grid, smem, st);
}
}  // namespace pkvd
