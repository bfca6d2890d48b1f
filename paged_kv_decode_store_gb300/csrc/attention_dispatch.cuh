// Per-dtype instantiation of the partition kernel for every supported
// (head_dim, heads-per-warp, group bound, path) combination.  Each dtype
// lives in its own translation unit so the build compiles them in parallel.
#pragma once

#include "attention_kernels.cuh"

namespace pkvd {

template <typename T, int D, int HPW>
cudaError_t dispatch_fma_g(const PartParams& pp, int gmax, int grid, size_t smem, cudaStream_t st) {
  switch (gmax) {
    case 1: return launch_partition<T, D, FmaConsumer<T, D, HPW, 1>>(pp, grid, smem, st);
    case 2: return launch_partition<T, D, FmaConsumer<T, D, HPW, 2>>(pp, grid, smem, st);
    case 4: return launch_partition<T, D, FmaConsumer<T, D, HPW, 4>>(pp, grid, smem, st);
    default: return launch_partition<T, D, FmaConsumer<T, D, HPW, 8>>(pp, grid, smem, st);
  }
}

template <typename T, int D>
cudaError_t dispatch_d(const PartParams& pp, int hpw, int gmax, int path, int grid, size_t smem,
                       cudaStream_t st) {
  if constexpr (sizeof(T) == 2) {
    if (path == PKVD_PATH_MMA) {
      return hpw == 1 ? launch_partition<T, D, MmaConsumer<T, D, 1>>(pp, grid, smem, st)
                      : launch_partition<T, D, MmaConsumer<T, D, 2>>(pp, grid, smem, st);
    }
    return hpw == 1 ? dispatch_fma_g<T, D, 1>(pp, gmax, grid, smem, st)
                    : dispatch_fma_g<T, D, 2>(pp, gmax, grid, smem, st);
  } else {
    if (path == PKVD_PATH_MMA || hpw != 1) return cudaErrorInvalidValue;
    return dispatch_fma_g<T, D, 1>(pp, gmax, grid, smem, st);
  }
}

template <typename T>
cudaError_t dispatch_partition(const PartParams& pp, int D, int hpw, int gmax, int path, int grid,
                               size_t smem, cudaStream_t st) {
  return D == 64 ? dispatch_d<T, 64>(pp, hpw, gmax, path, grid, smem, st)
                 : dispatch_d<T, 128>(pp, hpw, gmax, path, grid, smem, st);
}

cudaError_t partition_f32(const PartParams&, int, int, int, int, int, size_t, cudaStream_t);
cudaError_t partition_f16(const PartParams&, int, int, int, int, int, size_t, cudaStream_t);
cudaError_t partition_bf16(const PartParams&, int, int, int, int, int, size_t, cudaStream_t);

}  // namespace pkvd
