// Slot mapping and the paged KV-cache store (separately, or fused into one
// kernel for callers that need no slot mapping in between).
//
// nano-vllm "Model Runner" notes, sections "prefill and decode" and
// "allocated kv cache": the token decoded now is position context_len - 1;
// it lives in physical block block_table[pos / block_size] at row
// pos % block_size, i.e. slot = physical * block_size + pos % block_size,
// and its K and V rows are written there in place (the donated-buffer
// update of Grok-1 "第 8 章 runners.py 推理引擎", section 8.4).
//
// Both kernels are latency bound (a few KB per step): one warp-sized pass
// over rows, 16-byte vector copies, 64-bit cache offsets.
#include "common.cuh"
#include "launch.h"

namespace pkvd {

// Slot of row i's newest token, or -1 (empty row or a bad length / block id,
// which is flagged).
__device__ __forceinline__ int64_t decode_slot(const int32_t* __restrict__ tables, int max_blocks,
                                               const int32_t* __restrict__ ctx, int i, int block_size,
                                               int64_t num_blocks, int32_t* err) {
  const int c = ctx[i];
  if (c < 0) {
    flag_error(err, PKVD_ERR_CONTEXT);
    return -1;
  }
  if (c == 0) return -1;
  const int pos = c - 1;
  const int logical = pos / block_size;
  if (logical >= max_blocks) {
    flag_error(err, PKVD_ERR_CONTEXT);
    return -1;
  }
  const int phys = tables[(int64_t)i * max_blocks + logical];
  if (phys < 0 || phys >= num_blocks) {
    flag_error(err, PKVD_ERR_BLOCK_ID);
    return -1;
  }
  return (int64_t)phys * block_size + pos % block_size;
}

__global__ void slot_mapping_kernel(int64_t* __restrict__ slots, const int32_t* __restrict__ tables,
                                    int max_blocks, const int32_t* __restrict__ ctx, int num_seqs,
                                    int block_size, int64_t num_blocks, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= num_seqs) return;
  slots[i] = decode_slot(tables, max_blocks, ctx, i, block_size, num_blocks, err);
}

// Copy token tok's K and V rows (num_heads x head_dim each, 16-byte
// vectors, threads striding) to cache slot `slot`.  Element e of a row is
// (head e / D, dim e % D).
__device__ __forceinline__ void store_rows(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v, int tok,
                                           int64_t slot, uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                                           int block_size, int num_heads, int head_dim, int64_t block_stride,
                                           int64_t token_stride, int64_t head_stride, int elem_bytes) {
  const int64_t blk = slot / block_size;
  const int64_t row = slot % block_size;
  const int64_t base = blk * block_stride + row * token_stride;   // elements
  const int vec_elems = 16 / elem_bytes;
  const int row_elems = num_heads * head_dim;
  const int nvec = row_elems / vec_elems;
  const uint4* ksrc = reinterpret_cast<const uint4*>(k + (int64_t)tok * row_elems * elem_bytes);
  const uint4* vsrc = reinterpret_cast<const uint4*>(v + (int64_t)tok * row_elems * elem_bytes);
  for (int idx = threadIdx.x; idx < 2 * nvec; idx += blockDim.x) {
    const int which = idx >= nvec;
    const int vi = which ? idx - nvec : idx;
    const int e = vi * vec_elems;
    const int h = e / head_dim, d = e % head_dim;
    const int64_t off = (base + h * head_stride + d) * elem_bytes;
    const uint4 val = which ? __ldg(vsrc + vi) : __ldg(ksrc + vi);
    *reinterpret_cast<uint4*>((which ? vc : kc) + off) = val;
  }
}

// One CTA per token row, the slot from a slot mapping.
__global__ void kv_store_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                const int64_t* __restrict__ slots, uint8_t* __restrict__ kc,
                                uint8_t* __restrict__ vc, int64_t num_blocks, int block_size,
                                int num_heads, int head_dim, int64_t block_stride,
                                int64_t token_stride, int64_t head_stride, int elem_bytes,
                                int32_t* err) {
  pdl_trigger();
  pdl_wait();                       // slots come from the slot-mapping kernel
  const int tok = blockIdx.x;
  const int64_t slot = slots[tok];
  if (slot < 0) return;
  if (slot >= num_blocks * block_size) {
    if (threadIdx.x == 0) flag_error(err, PKVD_ERR_SLOT);
    return;
  }
  store_rows(k, v, tok, slot, kc, vc, block_size, num_heads, head_dim, block_stride, token_stride, head_stride,
             elem_bytes);
}

// Slot mapping and store in one kernel: one CTA per row computes its slot
// from the block table (every thread, the same two loads), optionally
// records it, and copies the rows.
__global__ void kv_store_paged_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                      const int32_t* __restrict__ tables, int max_blocks,
                                      const int32_t* __restrict__ ctx, int64_t* __restrict__ slots_out,
                                      uint8_t* __restrict__ kc, uint8_t* __restrict__ vc, int64_t num_blocks,
                                      int block_size, int num_heads, int head_dim, int64_t block_stride,
                                      int64_t token_stride, int64_t head_stride, int elem_bytes, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int tok = blockIdx.x;
  const int64_t slot = decode_slot(tables, max_blocks, ctx, tok, block_size, num_blocks,
                                   threadIdx.x == 0 ? err : nullptr);
  if (slots_out && threadIdx.x == 0) slots_out[tok] = slot;
  if (slot < 0) return;
  store_rows(k, v, tok, slot, kc, vc, block_size, num_heads, head_dim, block_stride, token_stride, head_stride,
             elem_bytes);
}

// Slot of new token row t of a varlen prefill batch, or -1 (a row past
// cu_seqlens_q[num_seqs], or a bad length / block id, which is flagged).
// nano-vllm "Model Runner" notes, section "prefix cache": sequence i owns
// rows [cu_q[i], cu_q[i+1]) and k_len = cu_k[i+1] - cu_k[i] tokens in all,
// so row t sits at position (k_len - q_len) + (t - cu_q[i]).
__device__ __forceinline__ int64_t prefill_slot(const int32_t* __restrict__ tables, int max_blocks,
                                                const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k,
                                                int num_seqs, int t, int block_size, int64_t num_blocks,
                                                int32_t* err) {
  if (t >= cu_q[num_seqs]) return -1;
  int lo = 0, hi = num_seqs - 1;   // the last i with cu_q[i] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_q[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int q0 = cu_q[lo], q1 = cu_q[lo + 1];
  const int qlen = q1 - q0, klen = cu_k[lo + 1] - cu_k[lo];
  if (t < q0 || t >= q1 || klen < qlen) {
    flag_error(err, PKVD_ERR_CONTEXT);
    return -1;
  }
  const int pos = klen - qlen + (t - q0);
  const int logical = pos / block_size;
  if (logical >= max_blocks) {
    flag_error(err, PKVD_ERR_CONTEXT);
    return -1;
  }
  const int phys = tables[(int64_t)lo * max_blocks + logical];
  if (phys < 0 || phys >= num_blocks) {
    flag_error(err, PKVD_ERR_BLOCK_ID);
    return -1;
  }
  return (int64_t)phys * block_size + pos % block_size;
}

// Prefill store: one CTA per new token row finds its sequence and position,
// optionally records the slot and copies the K and V rows there.
__global__ void kv_store_prefill_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                        const int32_t* __restrict__ tables, int max_blocks,
                                        const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k,
                                        int num_seqs, int64_t* __restrict__ slots_out, uint8_t* __restrict__ kc,
                                        uint8_t* __restrict__ vc, int64_t num_blocks, int block_size,
                                        int num_heads, int head_dim, int64_t block_stride, int64_t token_stride,
                                        int64_t head_stride, int elem_bytes, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int tok = blockIdx.x;
  const int64_t slot = prefill_slot(tables, max_blocks, cu_q, cu_k, num_seqs, tok, block_size, num_blocks,
                                    threadIdx.x == 0 ? err : nullptr);
  if (slots_out && threadIdx.x == 0) slots_out[tok] = slot;
  if (slot < 0) return;
  store_rows(k, v, tok, slot, kc, vc, block_size, num_heads, head_dim, block_stride, token_stride, head_stride,
             elem_bytes);
}

cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* tables, int max_blocks,
                                const int32_t* ctx, int num_seqs, int block_size,
                                int64_t num_blocks, cudaStream_t stream, int32_t* err) {
  if (num_seqs == 0) return cudaSuccess;
  const int threads = 128;
  return launch_pdl(slot_mapping_kernel, dim3((num_seqs + threads - 1) / threads), dim3(threads), 0, stream, slots,
                    tables, max_blocks, ctx, num_seqs, block_size, num_blocks, err);
}

cudaError_t launch_kv_store(const void* k, const void* v, const int64_t* slots, int num_tokens,
                            const pkvd_cache& c, int elem_bytes, cudaStream_t stream,
                            int32_t* err) {
  if (num_tokens == 0) return cudaSuccess;
  const int nvec = c.num_kv_heads * c.head_dim * elem_bytes / 16;
  int threads = 2 * nvec;
  threads = threads < 64 ? 64 : (threads > 256 ? 256 : threads);
  return launch_pdl(kv_store_kernel, dim3(num_tokens), dim3(threads), 0, stream, static_cast<const uint8_t*>(k),
                    static_cast<const uint8_t*>(v), slots, static_cast<uint8_t*>(c.k_base),
                    static_cast<uint8_t*>(c.v_base), c.num_blocks, c.block_size, c.num_kv_heads, c.head_dim,
                    c.block_stride, c.token_stride, c.head_stride, elem_bytes, err);
}

// Copy-on-write of shared blocks: CTA (i, kv) copies the first rows[i]
// token rows of block src[i] to block dst[i] in the K (kv = 0) or V cache,
// 16-byte vectors over every head of each row.
__global__ void copy_blocks_kernel(uint8_t* __restrict__ kc, uint8_t* __restrict__ vc, const int32_t* __restrict__ src,
                                   const int32_t* __restrict__ dst, const int32_t* __restrict__ rows,
                                   int64_t num_blocks, int block_size, int num_heads, int head_dim,
                                   int64_t block_stride, int64_t token_stride, int64_t head_stride, int elem_bytes,
                                   int32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int s = src[i], d = dst[i], n = rows[i];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks || n < 0 || n > block_size) {
    if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(err, PKVD_ERR_BLOCK_ID);
    return;
  }
  uint8_t* base = blockIdx.y ? vc : kc;
  const int vec_elems = 16 / elem_bytes;
  const int per_head = head_dim / vec_elems;
  const int per_row = num_heads * per_head;
  for (int idx = threadIdx.x; idx < n * per_row; idx += blockDim.x) {
    const int t = idx / per_row, rem = idx % per_row;
    const int h = rem / per_head, c = rem % per_head;
    const int64_t off = ((int64_t)t * token_stride + (int64_t)h * head_stride + (int64_t)c * vec_elems) * elem_bytes;
    const uint4 val = *reinterpret_cast<const uint4*>(base + (int64_t)s * block_stride * elem_bytes + off);
    *reinterpret_cast<uint4*>(base + (int64_t)d * block_stride * elem_bytes + off) = val;
  }
}

cudaError_t launch_copy_blocks(const pkvd_cache& c, int elem_bytes, const int32_t* src, const int32_t* dst,
                               const int32_t* rows, int count, cudaStream_t stream, int32_t* err) {
  if (count == 0) return cudaSuccess;
  return launch_pdl(copy_blocks_kernel, dim3(count, 2), dim3(256), 0, stream, static_cast<uint8_t*>(c.k_base),
                    static_cast<uint8_t*>(c.v_base), src, dst, rows, c.num_blocks, c.block_size, c.num_kv_heads,
                    c.head_dim, c.block_stride, c.token_stride, c.head_stride, elem_bytes, err);
}

cudaError_t launch_kv_store_paged(const void* k, const void* v, const int32_t* tables, int max_blocks,
                                  const int32_t* ctx, int num_seqs, int64_t* slots_out, const pkvd_cache& c,
                                  int elem_bytes, cudaStream_t stream, int32_t* err) {
  if (num_seqs == 0) return cudaSuccess;
  const int nvec = c.num_kv_heads * c.head_dim * elem_bytes / 16;
  int threads = 2 * nvec;
  threads = threads < 64 ? 64 : (threads > 256 ? 256 : threads);
  return launch_pdl(kv_store_paged_kernel, dim3(num_seqs), dim3(threads), 0, stream, static_cast<const uint8_t*>(k),
                    static_cast<const uint8_t*>(v), tables, max_blocks, ctx, slots_out,
                    static_cast<uint8_t*>(c.k_base), static_cast<uint8_t*>(c.v_base), c.num_blocks, c.block_size,
                    c.num_kv_heads, c.head_dim, c.block_stride, c.token_stride, c.head_stride, elem_bytes, err);
}

cudaError_t launch_kv_store_prefill(const void* k, const void* v, const int32_t* tables, int max_blocks,
                                    const int32_t* cu_q, const int32_t* cu_k, int num_seqs, int total_q,
                                    int64_t* slots_out, const pkvd_cache& c, int elem_bytes, cudaStream_t stream,
                                    int32_t* err) {
  if (total_q == 0) return cudaSuccess;
  const int nvec = c.num_kv_heads * c.head_dim * elem_bytes / 16;
  int threads = 2 * nvec;
  threads = threads < 64 ? 64 : (threads > 256 ? 256 : threads);
  return launch_pdl(kv_store_prefill_kernel, dim3(total_q), dim3(threads), 0, stream, static_cast<const uint8_t*>(k),
                    static_cast<const uint8_t*>(v), tables, max_blocks, cu_q, cu_k, num_seqs, slots_out,
                    static_cast<uint8_t*>(c.k_base), static_cast<uint8_t*>(c.v_base), c.num_blocks, c.block_size,
                    c.num_kv_heads, c.head_dim, c.block_stride, c.token_stride, c.head_stride, elem_bytes, err);
}

}  // namespace pkvd
