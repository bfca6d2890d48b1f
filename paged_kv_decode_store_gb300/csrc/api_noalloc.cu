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
// address is looked up with cudaGetSymbolAddress, once per device, by the
// first call on that device (with that device current).  Make that first
// call before any stream capture.
#include <atomic>

#include "launch.h"

namespace pkvd {

// 16 MiB.  The attention workspace grows with the partition grid (at most one
// CTA per SM) and the query heads, not with the rows: on a 152-SM GPU, 64
// query heads at head_dim 128 need 152 x 2 x 64 x 132 x 4 B = 10.3 MB, and
// 128 such heads (20.5 MB) are rejected.
constexpr size_t kNoAllocScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices] = {};   // set once per device

// Device address of the scratch on the current device (set-up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* ptr = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!ptr) {   // threads racing here all look up, and store, the same address
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev].store(ptr, std::memory_order_release);
  }
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
  // argument checks first, so a bad call never touches the device
  if (num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0) return PKVD_INVALID_ARG;
  if (!cache || cache->head_dim <= 0) return PKVD_INVALID_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return PKVD_CUDA_ERROR;
  const int grid = attention_grid(num_seqs, max_context_len, sms);
  const size_t need = attention_workspace_bytes(num_seqs, num_q_heads, cache->head_dim, grid);
  if (need > kNoAllocScratchBytes) return PKVD_WORKSPACE_TOO_SMALL;   // larger than the built-in scratch
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return PKVD_CUDA_ERROR;
  return pkvd_paged_decode_attention(out, q, cache, block_tables, max_blocks_per_seq, context_lens,
                                     max_context_len, num_seqs, num_q_heads, scale, scratch, need, stream,
                                     err_flag);
}

}  // extern "C"
