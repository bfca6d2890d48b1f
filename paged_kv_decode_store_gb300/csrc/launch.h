// Internal launchers shared between the kernel translation units and the
// C-ABI layer (api.cu).  Host-side argument validation happens in api.cu;
// these functions only size grids and enqueue kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkvd.h"

namespace pkvd {

// Decode-attention launch geometry shared by the workspace query and the
// launcher, so both derive the same grid.
constexpr int kChunk = 16;            // tokens per pipeline stage
constexpr int kConsumerWarps = 8;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;

struct AttnArgs {
  void* out;
  const void* q;
  const void* k_base;
  const void* v_base;
  int64_t block_stride, token_stride, head_stride;  // elements
  int64_t num_blocks;
  int block_size;
  int num_kv_heads;
  int num_q_heads;
  int head_dim;
  int dtype;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int max_context_len;
  int num_seqs;
  float scale;
  void* workspace;
  int32_t* err;
  int grid;           // partition CTAs
  int path;           // PKVD_PATH_FMA / PKVD_PATH_MMA (resolved)
  int window;         // > 0: sliding window of the newest `window` positions
};

int attention_grid(int num_seqs, int max_context_len, int sm_count);
size_t attention_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int grid);
bool attention_path_supported(int path, int dtype, int head_dim, int num_kv_heads, int group);
int attention_default_path(int dtype, int head_dim, int num_kv_heads, int group);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);
// Rows sharing their first prefix_len cached tokens (attention_prefix.cu):
// whether the shared-prefix kernel takes such a call, its workspace, and the
// launch (partition + merge).
bool prefix_path_usable(int dtype, int head_dim, int num_kv_heads, int num_q_heads, int num_seqs, int grid,
                        int prefix_len, int window);
size_t prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int grid,
                              int prefix_len);
cudaError_t launch_attention_prefix(const AttnArgs& a, int prefix_len, cudaStream_t stream);
// Host-side checks of a decode attention call (api.cu), shared by every
// attention entry point: resolves PKVD_PATH_AUTO in *path and, for a call
// with rows, gives the partition grid and the workspace bytes it needs.
// Checks nothing about the workspace itself.
pkvd_status attention_validate(void* out, const void* q, const pkvd_cache* cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len,
                               int32_t num_seqs, int32_t num_q_heads, float scale, int32_t window, int32_t* path,
                               int* grid, size_t* need);

cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* tables, int max_blocks,
                                const int32_t* ctx, int num_seqs, int block_size,
                                int64_t num_blocks, cudaStream_t stream, int32_t* err);

cudaError_t launch_kv_store(const void* k, const void* v, const int64_t* slots, int num_tokens,
                            const pkvd_cache& c, int elem_bytes, cudaStream_t stream,
                            int32_t* err);
cudaError_t launch_kv_store_paged(const void* k, const void* v, const int32_t* tables, int max_blocks,
                                  const int32_t* ctx, int num_seqs, int64_t* slots_out, const pkvd_cache& c,
                                  int elem_bytes, cudaStream_t stream, int32_t* err);
cudaError_t launch_copy_blocks(const pkvd_cache& c, int elem_bytes, const int32_t* src, const int32_t* dst,
                               const int32_t* rows, int count, cudaStream_t stream, int32_t* err);

// Varlen paged prefill (prefill.cu, store.cu).
struct PrefillArgs {
  void* out;
  const void* q;
  pkvd_cache cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int num_seqs;
  int total_q;
  int max_seqlen_q;
  int num_q_heads;
  float scale;
  int window;
  int32_t* err;
};
bool prefill_supported(int dtype, int head_dim, int group);
bool prefill_tc_supported(const PrefillArgs& a);
bool prefill_fma_supported(int dtype, int head_dim, int group, int num_kv_heads);
cudaError_t launch_prefill_fma(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream);
int prefill_tile_tokens(int group);
cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_kv_store_prefill(const void* k, const void* v, const int32_t* tables, int max_blocks,
                                    const int32_t* cu_q, const int32_t* cu_k, int num_seqs, int total_q,
                                    int64_t* slots_out, const pkvd_cache& c, int elem_bytes, cudaStream_t stream,
                                    int32_t* err);

// Per-row cut parameters the sampler leaves for the extras kernel:
// [0] flags (kRowGreedy, kRowUniform, kRowTopK), [1] nucleus threshold key
// (0 = off), [2] k-th key, [3] index of the last kept id at the k-th key
// (INT_MAX: every one), [4] the row max value (f32 bits), [5..7] unused.
constexpr int kRowInfo = 8;
constexpr int kRowGreedy = 1, kRowUniform = 2, kRowTopK = 4;

// One sampler call's arguments, for the two builds of the sampler kernel
// (sampler.cu: 1024-thread CTAs; sampler512.cu: 512-thread CTAs).
struct SampleCall {
  int32_t* token_ids;
  const void* logits;
  int dtype;
  int num_rows;
  int vocab;
  int64_t row_stride;
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const uint64_t* seeds;
  const uint64_t* offsets;
  const uint32_t* mask;
  int64_t mask_stride;
  int32_t* row_info;
};
// Each build: launch (or, with waves_only, only report how many waves of
// clusters it would need), and whether a masked row fits on chip.
namespace s1024 {
cudaError_t sample_launch(const SampleCall& c, cudaStream_t stream, int* waves_only);
bool sample_mask_fits(int dtype, int vocab, int64_t row_stride, const void* logits);
}  // namespace s1024
namespace s512 {
cudaError_t sample_launch(const SampleCall& c, cudaStream_t stream, int* waves_only);
bool sample_mask_fits(int dtype, int vocab, int64_t row_stride, const void* logits);
}  // namespace s512

cudaError_t launch_sample(int32_t* token_ids, const void* logits, int dtype, int num_rows,
                          int vocab, int64_t row_stride, const float* temperature,
                          const int32_t* top_k, const float* top_p, const uint64_t* seeds,
                          const uint64_t* offsets, const uint32_t* mask, int64_t mask_stride,
                          int32_t* row_info, cudaStream_t stream);
bool sample_mask_supported(int dtype, int vocab, int64_t row_stride, const void* logits);
cudaError_t launch_sample_extras(const void* logits, int dtype, int num_rows, int vocab, int64_t row_stride,
                                 const float* temperature, const uint32_t* mask, int64_t mask_stride,
                                 const int32_t* row_info, const int32_t* token_ids, float* token_prob,
                                 float* top_probs, int32_t* top_ids, cudaStream_t stream);

int device_sm_count();   // current device, cached; <= 0 on failure
int64_t device_l2_bytes();   // current device's L2 size in bytes, cached; 0 on failure

}  // namespace pkvd
