// The C ABI (include/pkvd.h): host-side argument checks, then one launcher
// call per entry point.  Nothing here allocates, synchronises or keeps state
// beyond per-device memos of the SM count and L2 size.
#include <cmath>

#include "device_cache.h"
#include "launch.h"

namespace pkvd {

namespace {
PerDeviceMemo<int> g_sm_count;
PerDeviceMemo<int64_t> g_l2_bytes;
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  const int known = g_sm_count.get(dev);
  if (known > 0) return known;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  g_sm_count.put(dev, n);
  return n;
}

int64_t device_l2_bytes() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  const int64_t known = g_l2_bytes.get(dev);
  if (known > 0) return known;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
  g_l2_bytes.put(dev, n);
  return n;
}

}  // namespace pkvd

using namespace pkvd;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int esize(int dtype) { return dtype == PKVD_F32 ? 4 : 2; }

bool valid_dtype(int dtype) { return dtype == PKVD_F32 || dtype == PKVD_F16 || dtype == PKVD_BF16; }

bool pow2(long long x) { return x > 0 && (x & (x - 1)) == 0; }

// Shared checks of a cache descriptor; `for_attention` adds the layout rules
// the bulk-copy pipeline needs.
pkvd_status check_cache(const pkvd_cache* c, bool for_attention) {
  if (!c || !c->k_base || !c->v_base) return PKVD_INVALID_ARG;
  if (!valid_dtype(c->dtype)) return PKVD_UNSUPPORTED_DTYPE;
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0 || c->block_size <= 0)
    return PKVD_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return PKVD_UNSUPPORTED_SHAPE;
  if (!pow2(c->block_size)) return PKVD_UNSUPPORTED_SHAPE;
  if (for_attention && c->block_size < 16) return PKVD_UNSUPPORTED_SHAPE;
  if (c->block_stride <= 0 || c->token_stride <= 0 || c->head_stride < c->head_dim)
    return PKVD_INVALID_ARG;
  const int e = esize(c->dtype);
  if (!aligned16(c->k_base) || !aligned16(c->v_base)) return PKVD_UNSUPPORTED_SHAPE;
  if ((c->block_stride * e) % 16 || (c->token_stride * e) % 16 || (c->head_stride * e) % 16)
    return PKVD_UNSUPPORTED_SHAPE;
  return PKVD_OK;
}

pkvd_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PKVD_OK : PKVD_CUDA_ERROR; }

}  // namespace

extern "C" {

const char* pkvd_status_string(pkvd_status s) {
  switch (s) {
    case PKVD_OK: return "ok";
    case PKVD_INVALID_ARG: return "invalid argument";
    case PKVD_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case PKVD_UNSUPPORTED_SHAPE: return "unsupported shape or alignment";
    case PKVD_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PKVD_CUDA_ERROR: return "CUDA runtime error";
    case PKVD_NO_SPACE: return "no free block";
  }
  return "unknown status";
}

int32_t pkvd_version(void) { return 100; }

pkvd_status pkvd_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs, int32_t block_size,
                              int64_t num_blocks, void* stream, int32_t* err_flag) {
  if (num_seqs < 0 || block_size <= 0 || num_blocks <= 0) return PKVD_INVALID_ARG;
  if (num_seqs == 0) return PKVD_OK;
  if (!slot_mapping || !block_tables || !context_lens || max_blocks_per_seq <= 0) return PKVD_INVALID_ARG;
  return from_cuda(launch_slot_mapping(slot_mapping, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                       block_size, num_blocks, static_cast<cudaStream_t>(stream), err_flag));
}

pkvd_status pkvd_kv_store(const void* k, const void* v, const int64_t* slot_mapping, int32_t num_tokens,
                          const pkvd_cache* cache, void* stream, int32_t* err_flag) {
  if (num_tokens < 0) return PKVD_INVALID_ARG;
  const pkvd_status cs = check_cache(cache, false);
  if (cs != PKVD_OK) return cs;
  if (num_tokens == 0) return PKVD_OK;
  if (!k || !v || !slot_mapping) return PKVD_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return PKVD_UNSUPPORTED_SHAPE;
  return from_cuda(launch_kv_store(k, v, slot_mapping, num_tokens, *cache, esize(cache->dtype),
                                   static_cast<cudaStream_t>(stream), err_flag));
}

pkvd_status pkvd_kv_store_paged(const void* k, const void* v, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                int64_t* slot_mapping, const pkvd_cache* cache, void* stream,
                                int32_t* err_flag) {
  if (num_seqs < 0) return PKVD_INVALID_ARG;
  const pkvd_status cs = check_cache(cache, false);
  if (cs != PKVD_OK) return cs;
  if (num_seqs == 0) return PKVD_OK;
  if (!k || !v || !block_tables || !context_lens || max_blocks_per_seq <= 0) return PKVD_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return PKVD_UNSUPPORTED_SHAPE;
  return from_cuda(launch_kv_store_paged(k, v, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                         slot_mapping, *cache, esize(cache->dtype),
                                         static_cast<cudaStream_t>(stream), err_flag));
}

pkvd_status pkvd_copy_blocks(const pkvd_cache* cache, const int32_t* src, const int32_t* dst, const int32_t* rows,
                             int32_t count, void* stream, int32_t* err_flag) {
  if (count < 0) return PKVD_INVALID_ARG;
  const pkvd_status cs = check_cache(cache, false);
  if (cs != PKVD_OK) return cs;
  if (count == 0) return PKVD_OK;
  if (!src || !dst || !rows) return PKVD_INVALID_ARG;
  return from_cuda(launch_copy_blocks(*cache, esize(cache->dtype), src, dst, rows, count,
                                      static_cast<cudaStream_t>(stream), err_flag));
}

pkvd_status pkvd_kv_store_prefill(const void* k, const void* v, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                                  const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                                  int64_t* slot_mapping, const pkvd_cache* cache, void* stream,
                                  int32_t* err_flag) {
  if (num_seqs < 0 || total_q < 0) return PKVD_INVALID_ARG;
  const pkvd_status cs = check_cache(cache, false);
  if (cs != PKVD_OK) return cs;
  if (total_q == 0) return PKVD_OK;
  if (!k || !v || !cu_seqlens_q || !cu_seqlens_k) return PKVD_INVALID_ARG;
  if (num_seqs > 0 && (!block_tables || max_blocks_per_seq <= 0)) return PKVD_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return PKVD_UNSUPPORTED_SHAPE;
  return from_cuda(launch_kv_store_prefill(k, v, block_tables, max_blocks_per_seq, cu_seqlens_q, cu_seqlens_k,
                                           num_seqs, total_q, slot_mapping, *cache, esize(cache->dtype),
                                           static_cast<cudaStream_t>(stream), err_flag));
}

pkvd_status pkvd_prefill_attention_ex(void* out, const void* q, const pkvd_cache* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                                      const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                                      int32_t max_seqlen_q, int32_t num_q_heads, float scale, int32_t window,
                                      void* stream, int32_t* err_flag, int32_t path) {
  if (path != PKVD_PATH_AUTO && path != PKVD_PATH_MMA && path != PKVD_PATH_TC && path != PKVD_PATH_FMA)
    return PKVD_INVALID_ARG;
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || window < 0) return PKVD_INVALID_ARG;
  if (!std::isfinite(scale)) return PKVD_INVALID_ARG;
  const pkvd_status cs = check_cache(cache, false);
  if (cs != PKVD_OK) return cs;
  if (num_q_heads <= 0) return PKVD_INVALID_ARG;
  if (num_q_heads % cache->num_kv_heads) return PKVD_UNSUPPORTED_SHAPE;
  const int group = num_q_heads / cache->num_kv_heads;
  const bool mma = prefill_supported(cache->dtype, cache->head_dim, group);
  const bool fma = prefill_fma_supported(cache->dtype, cache->head_dim, group, cache->num_kv_heads);
  if ((path == PKVD_PATH_MMA || path == PKVD_PATH_TC) && !mma)
    return cache->dtype == PKVD_F32 ? PKVD_UNSUPPORTED_DTYPE : PKVD_UNSUPPORTED_SHAPE;
  if ((path == PKVD_PATH_FMA || path == PKVD_PATH_AUTO) && !fma && !mma) return PKVD_UNSUPPORTED_SHAPE;
  if (path == PKVD_PATH_FMA && !fma) return PKVD_UNSUPPORTED_SHAPE;
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PKVD_OK;
  if (!out || !q || !block_tables || !cu_seqlens_q || !cu_seqlens_k || max_blocks_per_seq <= 0)
    return PKVD_INVALID_ARG;
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(out) & 3u)) return PKVD_UNSUPPORTED_SHAPE;
  const int tiles = mma ? (max_seqlen_q + prefill_tile_tokens(group) - 1) / prefill_tile_tokens(group) : 0;
  if (num_seqs > 65535 || tiles > 65535) return PKVD_UNSUPPORTED_SHAPE;
  PrefillArgs a;
  a.out = out;
  a.q = q;
  a.cache = *cache;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.max_seqlen_q = max_seqlen_q;
  a.num_q_heads = num_q_heads;
  a.scale = scale;
  a.window = window;
  a.err = err_flag;
  const bool tc = mma && prefill_tc_supported(a);
  if (path == PKVD_PATH_TC && !tc) return PKVD_UNSUPPORTED_SHAPE;
  if (path == PKVD_PATH_AUTO) path = tc ? PKVD_PATH_TC : mma ? PKVD_PATH_MMA : PKVD_PATH_FMA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (path == PKVD_PATH_TC) return from_cuda(launch_prefill_tc(a, st));
  if (path == PKVD_PATH_MMA) return from_cuda(launch_prefill_attention(a, st));
  return from_cuda(launch_prefill_fma(a, st));
}

pkvd_status pkvd_prefill_attention(void* out, const void* q, const pkvd_cache* cache, const int32_t* block_tables,
                                   int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                                   int32_t max_seqlen_q, int32_t num_q_heads, float scale, int32_t window,
                                   void* stream, int32_t* err_flag) {
  return pkvd_prefill_attention_ex(out, q, cache, block_tables, max_blocks_per_seq, cu_seqlens_q, cu_seqlens_k,
                                   num_seqs, total_q, max_seqlen_q, num_q_heads, scale, window, stream, err_flag,
                                   PKVD_PATH_AUTO);
}

pkvd_status pkvd_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                        int32_t max_context_len, int32_t sm_count, size_t* bytes) {
  if (!bytes || num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0) return PKVD_INVALID_ARG;
  if (sm_count <= 0) sm_count = device_sm_count();
  if (sm_count <= 0) return PKVD_CUDA_ERROR;
  const int grid = attention_grid(num_seqs, max_context_len, sm_count);
  *bytes = attention_workspace_bytes(num_seqs, num_q_heads, head_dim, grid);
  return PKVD_OK;
}

}  // extern "C"

namespace pkvd {

pkvd_status attention_validate(void* out, const void* q, const pkvd_cache* cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len,
                               int32_t num_seqs, int32_t num_q_heads, float scale, int32_t window, int32_t* path,
                               int* grid, size_t* need) {
  *grid = 0;
  *need = 0;
  if (num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0 || !std::isfinite(scale)) return PKVD_INVALID_ARG;
  const pkvd_status cs = check_cache(cache, true);
  if (cs != PKVD_OK) return cs;
  if (num_q_heads % cache->num_kv_heads) return PKVD_UNSUPPORTED_SHAPE;
  const int G = num_q_heads / cache->num_kv_heads;
  if (*path == PKVD_PATH_AUTO) *path = attention_default_path(cache->dtype, cache->head_dim, cache->num_kv_heads, G);
  if (*path != PKVD_PATH_FMA && *path != PKVD_PATH_MMA) {
    if (*path == 0 || *path == PKVD_PATH_TC) return PKVD_UNSUPPORTED_SHAPE;
    return PKVD_INVALID_ARG;
  }
  if (!attention_path_supported(*path, cache->dtype, cache->head_dim, cache->num_kv_heads, G))
    return PKVD_UNSUPPORTED_SHAPE;
  if (num_seqs == 0) return PKVD_OK;
  if (!out || !q || !block_tables || !context_lens || max_blocks_per_seq <= 0) return PKVD_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q)) return PKVD_UNSUPPORTED_SHAPE;
  const int sms = device_sm_count();
  if (sms <= 0) return PKVD_CUDA_ERROR;
  // a window shortens every row's span: fewer units, never a larger grid
  const int span = (window > 0 && window < max_context_len) ? window : max_context_len;
  *grid = attention_grid(num_seqs, span, sms);
  *need = attention_workspace_bytes(num_seqs, num_q_heads, cache->head_dim, *grid);
  return PKVD_OK;
}

}  // namespace pkvd

extern "C" {

namespace {
AttnArgs attn_args(void* out, const void* q, const pkvd_cache* cache, const int32_t* block_tables,
                   int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len, int32_t num_seqs,
                   int32_t num_q_heads, float scale, int32_t window, void* workspace, int32_t* err_flag, int grid,
                   int32_t path) {
  AttnArgs a;
  a.out = out;
  a.q = q;
  a.k_base = cache->k_base;
  a.v_base = cache->v_base;
  a.block_stride = cache->block_stride;
  a.token_stride = cache->token_stride;
  a.head_stride = cache->head_stride;
  a.num_blocks = cache->num_blocks;
  a.block_size = cache->block_size;
  a.num_kv_heads = cache->num_kv_heads;
  a.num_q_heads = num_q_heads;
  a.head_dim = cache->head_dim;
  a.dtype = cache->dtype;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.max_context_len = max_context_len;
  a.num_seqs = num_seqs;
  a.scale = scale;
  a.workspace = workspace;
  a.err = err_flag;
  a.grid = grid;
  a.path = path;
  a.window = window > 0 ? window : 0;
  return a;
}

pkvd_status attention_call(void* out, const void* q, const pkvd_cache* cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len,
                           int32_t num_seqs, int32_t num_q_heads, float scale, int32_t window, void* workspace,
                           size_t workspace_bytes, void* stream, int32_t* err_flag, int32_t path) {
  int grid = 0;
  size_t need = 0;
  const pkvd_status vs = attention_validate(out, q, cache, block_tables, max_blocks_per_seq, context_lens,
                                            max_context_len, num_seqs, num_q_heads, scale, window, &path, &grid,
                                            &need);
  if (vs != PKVD_OK || num_seqs == 0) return vs;
  if (!workspace || workspace_bytes < need) return PKVD_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return PKVD_UNSUPPORTED_SHAPE;
  const AttnArgs a = attn_args(out, q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                               num_seqs, num_q_heads, scale, window, workspace, err_flag, grid, path);
  return from_cuda(launch_attention(a, static_cast<cudaStream_t>(stream)));
}
}  // namespace

pkvd_status pkvd_paged_decode_attention_ex(void* out, const void* q, const pkvd_cache* cache,
                                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, int32_t max_context_len,
                                           int32_t num_seqs, int32_t num_q_heads, float scale,
                                           void* workspace, size_t workspace_bytes, void* stream,
                                           int32_t* err_flag, int32_t path) {
  return attention_call(out, q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                        num_q_heads, scale, 0, workspace, workspace_bytes, stream, err_flag, path);
}

pkvd_status pkvd_paged_decode_attention_window(void* out, const void* q, const pkvd_cache* cache,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, int32_t max_context_len,
                                               int32_t num_seqs, int32_t num_q_heads, float scale, int32_t window,
                                               void* workspace, size_t workspace_bytes, void* stream,
                                               int32_t* err_flag, int32_t path) {
  if (window < 0) return PKVD_INVALID_ARG;
  return attention_call(out, q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                        num_q_heads, scale, window, workspace, workspace_bytes, stream, err_flag, path);
}

pkvd_status pkvd_decode_prefix_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t max_context_len, int32_t prefix_len,
                                               int32_t sm_count, size_t* bytes) {
  if (!bytes || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
      prefix_len < 0)
    return PKVD_INVALID_ARG;
  if (sm_count <= 0) sm_count = device_sm_count();
  if (sm_count <= 0) return PKVD_CUDA_ERROR;
  const int grid = attention_grid(num_seqs, max_context_len, sm_count);
  const size_t plain = attention_workspace_bytes(num_seqs, num_q_heads, head_dim, grid);
  const size_t pre = prefix_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, grid, prefix_len);
  *bytes = plain > pre ? plain : pre;
  return PKVD_OK;
}

pkvd_status pkvd_paged_decode_attention_prefix(void* out, const void* q, const pkvd_cache* cache,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, int32_t max_context_len,
                                               int32_t num_seqs, int32_t num_q_heads, float scale,
                                               int32_t prefix_len, void* workspace, size_t workspace_bytes,
                                               void* stream, int32_t* err_flag) {
  if (prefix_len < 0) return PKVD_INVALID_ARG;
  int32_t path = PKVD_PATH_AUTO;
  int grid = 0;
  size_t need = 0;
  const pkvd_status vs = attention_validate(out, q, cache, block_tables, max_blocks_per_seq, context_lens,
                                            max_context_len, num_seqs, num_q_heads, scale, 0, &path, &grid, &need);
  if (vs != PKVD_OK) return vs;
  if (prefix_len % cache->block_size) return PKVD_INVALID_ARG;      // whole blocks are shared
  if (num_seqs == 0) return PKVD_OK;
  const bool usable = path == PKVD_PATH_MMA && grid > 0 &&
                      prefix_path_usable(cache->dtype, cache->head_dim, cache->num_kv_heads, num_q_heads, num_seqs,
                                         grid, prefix_len, 0);
  if (!usable)   // the same result from the plain kernel
    return attention_call(out, q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                          num_q_heads, scale, 0, workspace, workspace_bytes, stream, err_flag, path);
  const size_t need_p = prefix_workspace_bytes(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, grid,
                                               prefix_len);
  if (!workspace || workspace_bytes < need_p) return PKVD_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return PKVD_UNSUPPORTED_SHAPE;
  const AttnArgs a = attn_args(out, q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                               num_seqs, num_q_heads, scale, 0, workspace, err_flag, grid, path);
  return from_cuda(launch_attention_prefix(a, prefix_len, static_cast<cudaStream_t>(stream)));
}

pkvd_status pkvd_paged_decode_attention(void* out, const void* q, const pkvd_cache* cache,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t max_context_len, int32_t num_seqs,
                                        int32_t num_q_heads, float scale, void* workspace, size_t workspace_bytes,
                                        void* stream, int32_t* err_flag) {
  return pkvd_paged_decode_attention_ex(out, q, cache, block_tables, max_blocks_per_seq, context_lens,
                                        max_context_len, num_seqs, num_q_heads, scale, workspace, workspace_bytes,
                                        stream, err_flag, PKVD_PATH_AUTO);
}

pkvd_status pkvd_sample_workspace_bytes(int32_t num_rows, int32_t vocab, size_t* bytes) {
  if (!bytes || num_rows < 0 || vocab <= 0) return PKVD_INVALID_ARG;
  *bytes = (size_t)num_rows * kRowInfo * sizeof(int32_t);     // per-row cut parameters (extras only)
  return PKVD_OK;
}

pkvd_status pkvd_sample_ex(int32_t* token_ids, const void* logits, int32_t dtype, int32_t num_rows, int32_t vocab,
                           int64_t row_stride, const float* temperature, const int32_t* top_k, const float* top_p,
                           const uint64_t* seeds, const uint64_t* offsets, const uint32_t* mask,
                           int64_t mask_words_per_row, float* token_prob, float* top_probs, int32_t* top_ids,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dtype(dtype)) return PKVD_UNSUPPORTED_DTYPE;
  if (num_rows < 0 || vocab <= 0 || row_stride < vocab) return PKVD_INVALID_ARG;
  if (vocab > (1 << 23)) return PKVD_UNSUPPORTED_SHAPE;
  if (mask && mask_words_per_row < ((int64_t)vocab + 31) / 32) return PKVD_INVALID_ARG;
  if (num_rows == 0) return PKVD_OK;
  if (!token_ids || !logits || !temperature || !top_k || !top_p || !seeds || !offsets) return PKVD_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % esize(dtype)) return PKVD_UNSUPPORTED_SHAPE;
  if (mask && (reinterpret_cast<uintptr_t>(mask) % 4 || !sample_mask_supported(dtype, vocab, row_stride, logits)))
    return PKVD_UNSUPPORTED_SHAPE;
  const bool extras = token_prob || top_probs || top_ids;
  int32_t* row_info = nullptr;
  if (extras) {
    size_t need = 0;
    pkvd_sample_workspace_bytes(num_rows, vocab, &need);
    if (!workspace || workspace_bytes < need) return PKVD_WORKSPACE_TOO_SMALL;
    if (reinterpret_cast<uintptr_t>(workspace) % 4) return PKVD_UNSUPPORTED_SHAPE;
    row_info = static_cast<int32_t*>(workspace);
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_sample(token_ids, logits, dtype, num_rows, vocab, row_stride, temperature, top_k, top_p,
                                seeds, offsets, mask, mask_words_per_row, row_info, st);
  if (e != cudaSuccess || !extras) return from_cuda(e);
  return from_cuda(launch_sample_extras(logits, dtype, num_rows, vocab, row_stride, temperature, mask,
                                        mask_words_per_row, row_info, token_ids, token_prob, top_probs, top_ids,
                                        st));
}

pkvd_status pkvd_sample(int32_t* token_ids, const void* logits, int32_t dtype, int32_t num_rows, int32_t vocab,
                        int64_t row_stride, const float* temperature, const int32_t* top_k, const float* top_p,
                        const uint64_t* seeds, const uint64_t* offsets, void* workspace, size_t workspace_bytes,
                        void* stream) {
  return pkvd_sample_ex(token_ids, logits, dtype, num_rows, vocab, row_stride, temperature, top_k, top_p, seeds,
                        offsets, nullptr, 0, nullptr, nullptr, nullptr, workspace, workspace_bytes, stream);
}

}  // extern "C"
