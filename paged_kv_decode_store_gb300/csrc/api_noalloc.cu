// pkvd_paged_decode_attention_noalloc: paged decode attention whose scratch
// lives in a fixed array inside this library instead of a caller-supplied
// workspace.
//
// For callers that cannot allocate device memory at the point of the call:
// engines that hand all free device memory to the paged KV cache at start-up
// (a later cudaMalloc fails or evicts cache blocks), plugins inside a runtime
// that owns every device allocation through its own pool, latency-critical
// loops where cudaMalloc/cudaFree would synchronise the device, and plain C
// hosts with no device allocator of their own.  They pass inputs and outputs
// only.
//
// The scratch is one file-scope device array of kNoAllocScratchBytes.  Every
// GPU that loads this library holds it until the process exits, and every
// call on that GPU shares it: calls that overlap on the GPU (different
// streams without ordering between them) race on it and give wrong results.
// Nothing in it has to start at zero: each call writes every merge record it
// later reads, so the previous call's contents do no harm.
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, with the call's device
// current, on every call made outside stream capture: the address belongs to
// the current context, which a cudaDeviceReset or a caller-made driver
// context replaces.  A call made while its stream is capturing reuses the
// address that the last uncaptured call on that device found (a lookup could
// load the module, which capture forbids), so make one uncaptured call on
// each device, in the context that will replay the graph, before capturing.
#include <atomic>

#include "device_cache.h"
#include "launch.h"

namespace pkvd {

// 16 MiB.  The attention workspace grows with the partition grid (at most one
// CTA per SM) and the query heads, not with the rows: on a 152-SM GPU, 64
// query heads at head_dim 128 need 152 x 2 x 64 x 132 x 4 B = 10.3 MB, and
// 128 such heads (20.5 MB) are rejected.
constexpr size_t kNoAllocScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// the address the last uncaptured call on each device found
PerDeviceMemo<uintptr_t> g_scratch_addr;

// Device address of the scratch in the current context.
cudaError_t scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  if (cap != cudaStreamCaptureStatusNone) {
    const uintptr_t known = g_scratch_addr.get(dev);
    if (known) {
      *out = reinterpret_cast<void*>(known);
      return cudaSuccess;
    }
  }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (cap == cudaStreamCaptureStatusNone) g_scratch_addr.put(dev, reinterpret_cast<uintptr_t>(ptr));
  *out = ptr;
  return cudaSuccess;
}
}  // namespace

}  // namespace pkvd

using namespace pkvd;

extern "C" {

pkvd_status pkvd_paged_decode_attention_noalloc(void* out, const void* q, const pkvd_cache* cache,
                                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                const int32_t* context_lens, int32_t max_context_len,
                                                int32_t num_seqs, int32_t num_q_heads, float scale, void* stream,
                                                int32_t* err_flag) {
  // the workspace entry point's own checks first, so every invalid call gets
  // the same status from both entry points and never touches the device
  int32_t path = PKVD_PATH_AUTO;
  int grid = 0;
  size_t need = 0;
  const pkvd_status vs = attention_validate(out, q, cache, block_tables, max_blocks_per_seq, context_lens,
                                            max_context_len, num_seqs, num_q_heads, scale, 0, &path, &grid, &need);
  if (vs != PKVD_OK || num_seqs == 0) return vs;
  if (need > kNoAllocScratchBytes) return PKVD_WORKSPACE_TOO_SMALL;   // larger than the built-in scratch
  void* scratch = nullptr;
  if (scratch_address(static_cast<cudaStream_t>(stream), &scratch) != cudaSuccess) return PKVD_CUDA_ERROR;
  return pkvd_paged_decode_attention(out, q, cache, block_tables, max_blocks_per_seq, context_lens,
                                     max_context_len, num_seqs, num_q_heads, scale, scratch, need, stream,
                                     err_flag);
}

}  // extern "C"
