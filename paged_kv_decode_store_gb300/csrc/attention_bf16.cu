// Partition-kernel instantiations for __nv_bfloat16 caches.
#include "attention_dispatch.cuh"

namespace pkvd {
cudaError_t partition_bf16(const PartParams& pp, int D, int hpw, int gmax, int path, int grid, size_t smem,
                         cudaStream_t st) {
  return dispatch_partition<__nv_bfloat16>(pp, D, hpw, gmax, path, grid, smem, st);
}
}  // namespace pkvd
