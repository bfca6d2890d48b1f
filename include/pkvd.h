/*
 * pkvd.h -- C ABI of the paged KV-cache decode step for GB300 (sm_103a).
 *
 * One decode step of a paged-KV inference engine, as the pages describe it:
 *
 *   slot mapping   nano-vllm "Model Runner" notes, sections "prefill and
 *                  decode" and "allocated kv cache" (slot = block_table
 *                  [pos / block_size] * block_size + pos % block_size, with
 *                  pos = context_len - 1 for the token decoded now).
 *   kv_store       same notes, "prepare Prefill" / "allocated kv cache": the
 *                  new token's K and V are written into its slot of the
 *                  per-layer cache, in place (Grok-1 "第 8 章 runners.py
 *                  推理引擎", section 8.4 donated buffers, section 8.5 cache
 *                  shapes and updates).
 *   attention      single-query grouped-query attention of the new token
 *                  over the sequence's block table up to context_len (same
 *                  notes, "prefill and decode"; Grok-1 section 8.5 GQA 48:8;
 *                  Grok-1 section 8.2.3: an inactive row, context 0, gives a
 *                  zero output).
 *   sample         temperature, top-k, nucleus cut, Gumbel-max draw (Grok-1
 *                  sections 8.3 and 8.3.1 sample_token / top_p_filter;
 *                  nanochat "04 · Engine" section 3 top-k; nano-vllm "run
 *                  model" Gumbel-max sampler).
 *
 * Around it: the varlen prefill store and causal attention over cached
 * prefixes (nano-vllm "prefix cache"), sliding-window decode attention
 * (nanochat "推理基准 infer_bench.py"), the rest of Grok-1's sample_token
 * (mask, token probability, top-8), and a host block manager with prefix
 * sharing and copy-on-write.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers unless stated; sizes are
 *     element counts; strides are in elements.  `stream` is a cudaStream_t
 *     (NULL = legacy default stream).  Every call only enqueues work on
 *     `stream` and returns; nothing synchronises, nothing allocates, no
 *     state is kept between calls.  The caller owns every buffer, including
 *     workspaces, and may capture the calls in a CUDA graph.  (Two
 *     exceptions: the host block manager below, an object the caller
 *     creates and destroys, touched by host calls only; and
 *     pkvd_paged_decode_attention_noalloc, which takes no workspace but
 *     uses a scratch array built into the library and remembers its device
 *     address for calls under capture.  Its own comment gives its rules; the
 *     sentences above on workspaces, state and graph capture do not cover
 *     it.)
 *   - Argument checks run on the host before anything is enqueued and return
 *     a status code; the library never aborts, exits or traps.
 *   - `err_flag`, where present, is an optional device int32.  Kernels OR
 *     PKVD_ERR_* bits into it when they meet a bad index in device data
 *     (e.g. a block id outside the pool) and skip the offending access.
 *     The caller zeroes it and reads it back when it wants to know.
 *   - dtype codes: PKVD_F32, PKVD_F16, PKVD_BF16.  q, the new K/V, the cache
 *     and the attention output share one dtype.
 *   - Kernels are launched as programmatic dependents of the previous work
 *     on the stream: they may start while a preceding kernel that signalled
 *     early completion (griddepcontrol.launch_dependents) still runs.  Before
 *     waiting for it they read only inputs that no kernel of this library
 *     writes (context lengths, block tables, q); everything else (the cache,
 *     slot_mapping, outputs, workspaces) comes after the wait.  A caller's
 *     own kernel that signals early must not write those inputs of the call
 *     that follows it.
 */
#ifndef PKVD_H
#define PKVD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKVD_OK = 0,
  PKVD_INVALID_ARG = 1,          /* null pointer, negative size, bad scale ... */
  PKVD_UNSUPPORTED_DTYPE = 2,
  PKVD_UNSUPPORTED_SHAPE = 3,    /* head_dim, group size, block size, alignment */
  PKVD_WORKSPACE_TOO_SMALL = 4,
  PKVD_CUDA_ERROR = 5,           /* a CUDA runtime call failed (launch, query) */
  PKVD_NO_SPACE = 6              /* block manager: not enough free blocks (nothing changed) */
} pkvd_status;

typedef enum { PKVD_F32 = 0, PKVD_F16 = 1, PKVD_BF16 = 2 } pkvd_dtype;

/* Bits kernels OR into *err_flag. */
#define PKVD_ERR_BLOCK_ID    1   /* block-table entry outside [0, num_blocks) */
#define PKVD_ERR_SLOT        2   /* slot >= num_blocks * block_size           */
#define PKVD_ERR_CONTEXT     4   /* context_len < 0 or > the stated bound     */
#define PKVD_ERR_TIMEOUT     8   /* a pipeline wait gave up (never expected)  */

/* Attention path selector for pkvd_paged_decode_attention_ex and
 * pkvd_prefill_attention_ex. */
typedef enum {
  PKVD_PATH_AUTO = 0,   /* the library's choice for the shape              */
  PKVD_PATH_FMA = 1,    /* fp32 CUDA-core dot products                     */
  PKVD_PATH_MMA = 2,    /* warp-level mma.sync m16n8k16 tensor-core path   */
  PKVD_PATH_TC = 3      /* tcgen05: TMA-fed operands, TMEM accumulators
                           (prefill only)                                  */
} pkvd_attn_path;

/*
 * One layer's K and V cache, described without a copy.
 *
 * Element (block b, row r, kv head h, dim d) of K sits at
 *   k_base + b*block_stride + r*token_stride + h*head_stride + d
 * (same for V at v_base).  For nano-vllm's tensor
 *   kv_cache[2, num_layers, num_blocks, block_size, num_kv_heads, head_dim]
 * ("allocated kv cache") layer l is k_base = &kv_cache[0, l, 0, 0, 0, 0],
 * v_base = &kv_cache[1, l, 0, 0, 0, 0], block_stride = block_size*H*D,
 * token_stride = H*D, head_stride = D.
 * Requirements: head_dim in {64, 128}; block_size a power of two (>= 16 for
 * the decode attention, >= 8 for the tcgen05 prefill path); head_dim
 * elements contiguous; base pointers and every stride times the
 * element size multiples of 16 bytes.
 */
typedef struct {
  void* k_base;
  void* v_base;
  int32_t dtype;          /* pkvd_dtype */
  int32_t block_size;
  int64_t num_blocks;
  int32_t num_kv_heads;
  int32_t head_dim;
  int64_t block_stride;
  int64_t token_stride;
  int64_t head_stride;
} pkvd_cache;

/* Human-readable text of a status code (static storage). */
const char* pkvd_status_string(pkvd_status s);

/* Library version, major*10000 + minor*100 + patch. */
int32_t pkvd_version(void);

/*
 * pkvd_slot_mapping -- slot of each row's new token.
 *   slot_mapping[i] = block_tables[i*max_blocks_per_seq + (ctx_i-1)/block_size]
 *                     * block_size + (ctx_i-1) % block_size,  ctx_i = context_lens[i]
 *   and -1 where ctx_i == 0 (an inactive row).
 * Inputs: block_tables int32 [num_seqs, max_blocks_per_seq] row-major;
 *         context_lens int32 [num_seqs] (includes the new token).
 * Output: slot_mapping int64 [num_seqs].
 * Device errors: a block id outside [0, num_blocks) or a context longer than
 * max_blocks_per_seq*block_size sets the matching bit and writes -1.
 */
pkvd_status pkvd_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* context_lens,
                              int32_t num_seqs, int32_t block_size, int64_t num_blocks,
                              void* stream, int32_t* err_flag);

/*
 * pkvd_kv_store -- write each token's new K and V rows into its cache slot.
 *   K[slot / bs, slot % bs, :, :] = k[i, :, :];  V[...] = v[i, :, :]
 * an exact bit copy; rows with slot < 0 are skipped.
 * Inputs: k, v [num_tokens, num_kv_heads, head_dim] contiguous, cache dtype;
 *         slot_mapping int64 [num_tokens]; slots must be distinct.
 * Device errors: slot >= num_blocks*block_size sets PKVD_ERR_SLOT, row skipped.
 */
pkvd_status pkvd_kv_store(const void* k, const void* v, const int64_t* slot_mapping,
                          int32_t num_tokens, const pkvd_cache* cache, void* stream,
                          int32_t* err_flag);

/*
 * pkvd_kv_store_paged -- pkvd_slot_mapping and pkvd_kv_store in one kernel
 * (same passages as those two): row i's new K and V rows go to the slot of
 * its newest token, found from block_tables and context_lens as in
 * pkvd_slot_mapping, and the slot is also written to slot_mapping[i] when
 * slot_mapping is not NULL.  Rows with context_lens[i] == 0 are skipped
 * (slot -1).  One launch instead of two for a decode step that needs the
 * slots nowhere else.
 * Inputs: k, v [num_seqs, num_kv_heads, head_dim] contiguous, cache dtype,
 *         16-byte aligned; block_tables int32 [num_seqs, max_blocks_per_seq];
 *         context_lens int32 [num_seqs] (include the new token).
 * Output: the cache rows; slot_mapping int64 [num_seqs] or NULL.
 * Device errors: as pkvd_slot_mapping (bad block id or length: row skipped).
 */
pkvd_status pkvd_kv_store_paged(const void* k, const void* v, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* context_lens,
                                int32_t num_seqs, int64_t* slot_mapping, const pkvd_cache* cache,
                                void* stream, int32_t* err_flag);

/*
 * Workspace bytes pkvd_paged_decode_attention needs for these sizes on a
 * GPU with `sm_count` SMs (sm_count <= 0: query the current device).
 * Host only; returns PKVD_CUDA_ERROR if the device query fails.
 */
pkvd_status pkvd_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                        int32_t head_dim, int32_t max_context_len,
                                        int32_t sm_count, size_t* bytes);

/*
 * pkvd_paged_decode_attention -- one query token per sequence attends to
 * its cached context.  For row i, query head h, kv head hk = h / G
 * (G = num_q_heads / num_kv_heads, contiguous groups):
 *   s_j = scale * <q[i,h,:], K_j>,  j < context_lens[i],
 *   K_j = K[block_tables[i][j / bs], j % bs, hk, :]   (V_j likewise)
 *   out[i,h,:] = sum_j softmax(s)_j V_j ;  zeros when context_lens[i] == 0.
 * Inputs: q [num_seqs, num_q_heads, head_dim] contiguous, cache dtype;
 *         block_tables int32 [num_seqs, max_blocks_per_seq]; context_lens
 *         int32 [num_seqs], each <= max_context_len (a host-side bound used
 *         for the launch shape; larger values set PKVD_ERR_CONTEXT and are
 *         clamped).  Entries past a row's last block and cache rows past its
 *         context are never read.
 * Output: out [num_seqs, num_q_heads, head_dim], cache dtype, fp32 softmax
 *         and accumulation.
 * workspace: device scratch of at least pkvd_decode_workspace_bytes(...)
 *         bytes (16-byte aligned), used for split-context partial results;
 *         its contents need no initialisation.  Calls that share a
 *         workspace must not overlap on the GPU.
 * Requirements: num_q_heads % num_kv_heads == 0, group size <= 8,
 *         num_kv_heads <= 8 or == 16.
 */
pkvd_status pkvd_paged_decode_attention(void* out, const void* q, const pkvd_cache* cache,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t max_context_len,
                                        int32_t num_seqs, int32_t num_q_heads, float scale,
                                        void* workspace, size_t workspace_bytes,
                                        void* stream, int32_t* err_flag);

/* Same as pkvd_paged_decode_attention with an explicit compute path
 * (pkvd_attn_path); PKVD_UNSUPPORTED_SHAPE if the path cannot run the shape. */
pkvd_status pkvd_paged_decode_attention_ex(void* out, const void* q, const pkvd_cache* cache,
                                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, int32_t max_context_len,
                                           int32_t num_seqs, int32_t num_q_heads, float scale,
                                           void* workspace, size_t workspace_bytes,
                                           void* stream, int32_t* err_flag, int32_t path);

/*
 * pkvd_paged_decode_attention_window -- the same attention over a sliding
 * window: with window > 0 row i attends to its newest `window` positions,
 * j in [max(0, context_lens[i] - window), context_lens[i]) (nanochat
 * "04 · Engine 推理与工具调用", section "推理基准 infer_bench.py": a window
 * layer reads min(context, window) K/V rows; the newest positions, the new
 * token included, is the reading taken).  window == 0: no window (same as
 * _ex); window < 0: PKVD_INVALID_ARG.  Cache rows before the window are never
 * read.  The workspace of pkvd_decode_workspace_bytes for max_context_len is
 * always large enough.
 */
pkvd_status pkvd_paged_decode_attention_window(void* out, const void* q, const pkvd_cache* cache,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, int32_t max_context_len,
                                               int32_t num_seqs, int32_t num_q_heads, float scale,
                                               int32_t window, void* workspace, size_t workspace_bytes,
                                               void* stream, int32_t* err_flag, int32_t path);

/*
 * pkvd_decode_prefix_workspace_bytes -- workspace bytes of
 * pkvd_paged_decode_attention_prefix for these sizes (never less than
 * pkvd_decode_workspace_bytes for the same call; sm_count <= 0: the current
 * device's).  Host only.
 */
pkvd_status pkvd_decode_prefix_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t max_context_len, int32_t prefix_len,
                                               int32_t sm_count, size_t* bytes);

/*
 * pkvd_paged_decode_attention_prefix -- the same attention as
 * pkvd_paged_decode_attention for a batch whose rows share their first
 * prefix_len cached tokens: nanochat "04 · Engine 推理与工具调用", sections
 * 2-3, prefills a prompt once and clones its cache N ways, so every row's
 * first prefix_len / block_size block-table entries name the same physical
 * blocks.  Those blocks are read once per group of up to 16 / G rows (G
 * query heads per KV head), every query of the group applied to each staged
 * tile, instead of once per row.
 * Requirements: prefix_len a multiple of block_size (0: no sharing); every
 *         row's context longer than prefix_len (the token decoded now is the
 *         row's own; a row that is not longer sets PKVD_ERR_CONTEXT and its
 *         output is undefined); the shared entries equal in every row's
 *         table (the prefix is read through row 0's table; this is not
 *         checked).
 * The shared-prefix kernel runs for 16-bit caches with 8 KV heads of 64 or
 * 128 (the tensor-core consumer), at least two rows and no more row groups
 * than partition CTAs; any other call gives the same result through the
 * plain kernel.  Workspace: pkvd_decode_prefix_workspace_bytes.  Same input
 * contract, status codes and device errors as pkvd_paged_decode_attention.
 */
pkvd_status pkvd_paged_decode_attention_prefix(void* out, const void* q, const pkvd_cache* cache,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, int32_t max_context_len,
                                               int32_t num_seqs, int32_t num_q_heads, float scale,
                                               int32_t prefix_len, void* workspace, size_t workspace_bytes,
                                               void* stream, int32_t* err_flag);

/*
 * pkvd_paged_decode_attention_noalloc -- the same attention as
 * pkvd_paged_decode_attention (same arguments without the workspace pair,
 * same results and errors), for callers that cannot allocate device memory
 * where they call it: engines that give all free device memory to the paged
 * KV cache at start-up (a later cudaMalloc fails), plugins inside a runtime
 * that owns every device allocation, latency-critical loops where
 * cudaMalloc/cudaFree would synchronise the device, plain C hosts without a
 * device allocator.  The pages describe no such entry point; it exists for
 * those callers only.
 *
 * Instead of a caller workspace it uses one 16 MiB scratch array built into
 * the library (held on every GPU that loads the library until the process
 * exits).  Shapes whose workspace (pkvd_decode_workspace_bytes) exceeds
 * 16 MiB are rejected with PKVD_WORKSPACE_TOO_SMALL before anything is
 * enqueued.  All calls on a GPU share the array: calls that overlap on the
 * GPU (unordered streams) race and give wrong results.  Each call writes
 * every part of the array it reads, so nothing needs clearing between
 * calls.  Every call made outside stream capture looks up the array's
 * device address (cudaGetSymbolAddress) in the current context, so a
 * cudaDeviceReset or a context the caller made with the driver API is
 * followed.  A call on a capturing stream reuses the address the last
 * uncaptured call on that device found: make one uncaptured call per
 * device, in the context that will replay the graph, before capturing.
 * Argument checks, and their status codes, are the workspace entry
 * point's; the 16 MiB limit is checked after them.
 * Nothing is allocated.
 */
pkvd_status pkvd_paged_decode_attention_noalloc(void* out, const void* q, const pkvd_cache* cache,
                                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                const int32_t* context_lens, int32_t max_context_len,
                                                int32_t num_seqs, int32_t num_q_heads, float scale,
                                                void* stream, int32_t* err_flag);

/*
 * pkvd_kv_store_prefill -- the store of a varlen prefill batch (nano-vllm
 * "Model Runner" notes, sections "prepare Prefill" and "prefix cache": the
 * block table is filled before the step, and the step writes every newly
 * scheduled token's K and V rows to the slot its position maps to).
 * Sequence i owns new rows [cu_seqlens_q[i], cu_seqlens_q[i+1]) and has
 * k_len_i = cu_seqlens_k[i+1] - cu_seqlens_k[i] tokens in all, the first
 * k_len_i - q_len_i of them already cached (a prefix-cache hit or an earlier
 * chunk); new row t of sequence i is position p = (k_len_i - q_len_i) +
 * (t - cu_seqlens_q[i]) and goes to slot
 *   block_tables[i][p / bs] * bs + p % bs,
 * also written to slot_mapping[t] when slot_mapping is not NULL.
 * Inputs: k, v [total_q, num_kv_heads, head_dim] contiguous, cache dtype,
 *         16-byte aligned; cu_seqlens_q, cu_seqlens_k int32 [num_seqs + 1]
 *         device arrays, non-decreasing, starting at 0; block_tables int32
 *         [num_seqs, max_blocks_per_seq].
 * Output: the cache rows; slot_mapping int64 [total_q] or NULL.
 * Device errors: rows t >= cu_seqlens_q[num_seqs] are skipped (slot -1);
 *         q_len > k_len or a position past the table sets PKVD_ERR_CONTEXT,
 *         a block id outside [0, num_blocks) PKVD_ERR_BLOCK_ID; such rows
 *         are skipped.
 */
pkvd_status pkvd_kv_store_prefill(const void* k, const void* v, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                                  const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                                  int64_t* slot_mapping, const pkvd_cache* cache, void* stream,
                                  int32_t* err_flag);

/*
 * pkvd_prefill_attention -- varlen causal attention of a prefill batch over
 * the paged cache (nano-vllm "Model Runner" notes, sections "prefix cache"
 * and "prefill and decode": cu_seqlens_q / cu_seqlens_k describe the batch,
 * cu_seqlens_k[-1] > cu_seqlens_q[-1] when prefixes are cached, and prefill
 * runs its own dense, compute-bound kernel).  New row t of sequence i at
 * position p (as in pkvd_kv_store_prefill), query head h, kv head
 * hk = h / G:
 *   s_j = scale * <q[t,h,:], K_j>,  ws(p) <= j <= p,
 *   K_j = K[block_tables[i][j / bs], j % bs, hk, :]   (V_j likewise)
 *   out[t,h,:] = sum_j softmax(s)_j V_j,
 * ws(p) = max(0, p + 1 - window) for window > 0, else 0.  The cache must
 * already hold positions 0 .. k_len_i - 1 (run pkvd_kv_store_prefill first
 * on the same stream).  Rows of the cache outside [ws, p] of some new token
 * are never read.
 * Inputs: q [total_q, num_q_heads, head_dim] contiguous, cache dtype,
 *         16-byte aligned; cu_seqlens_q, cu_seqlens_k, block_tables as in
 *         pkvd_kv_store_prefill; max_seqlen_q >= every q_len (host bound that
 *         sizes the grid).
 * Output: out [total_q, num_q_heads, head_dim], cache dtype, 4-byte
 *         aligned; rows t >= cu_seqlens_q[num_seqs] are not written.
 *         Tensor-core products with fp32 accumulation; the softmax weights
 *         are rounded to the cache dtype for the second product.
 * Requirements: head_dim 64 or 128, num_q_heads % num_kv_heads == 0,
 *         num_seqs <= 65535, window >= 0; f16 / bf16 caches with group size
 *         <= 128 run on the tensor cores, f32 caches (and 16-bit ones on
 *         request) on the CUDA cores with group size <= 16.
 * Device errors: q_len > k_len, cu_seqlens_q[i+1] > total_q, k_len past the
 *         table or q_len > max_seqlen_q set PKVD_ERR_CONTEXT (that
 *         sequence's rows, or in the last case its earliest rows, are not
 *         written); a bad block id sets PKVD_ERR_BLOCK_ID (its rows read as
 *         zeros).
 */
pkvd_status pkvd_prefill_attention(void* out, const void* q, const pkvd_cache* cache, const int32_t* block_tables,
                                   int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                                   int32_t max_seqlen_q, int32_t num_q_heads, float scale, int32_t window,
                                   void* stream, int32_t* err_flag);

/* Same as pkvd_prefill_attention with an explicit compute path:
 * PKVD_PATH_TC (tcgen05 MMAs on TMA-loaded 128-byte-swizzled tiles with TMEM
 * accumulators; 16-bit caches, needs block_size >= 8, 16-byte aligned q and
 * out, and a cache whose strides nest head < token < block), PKVD_PATH_MMA
 * (mma.sync, 16-bit caches), PKVD_PATH_FMA (fp32 CUDA-core arithmetic, any
 * cache dtype, group size <= 16), or PKVD_PATH_AUTO (TC when it can run the
 * call, else MMA, else FMA; what pkvd_prefill_attention does).  PKVD_UNSUPPORTED_SHAPE if the path cannot
 * run the call.  Both paths compute the same function; on the TC path cache
 * rows of a 16-row-aligned group that meets a sequence's range may be
 * fetched, but rows outside [ws, p] never weigh in. */
pkvd_status pkvd_prefill_attention_ex(void* out, const void* q, const pkvd_cache* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                                      const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                                      int32_t max_seqlen_q, int32_t num_q_heads, float scale, int32_t window,
                                      void* stream, int32_t* err_flag, int32_t path);

/* Workspace bytes of pkvd_sample_ex's optional outputs: 32 per row (host
 * only).  pkvd_sample itself needs none (it may get NULL, 0). */
pkvd_status pkvd_sample_workspace_bytes(int32_t num_rows, int32_t vocab, size_t* bytes);

/*
 * pkvd_sample -- one token id per row of logits.
 * Row r (x = logits[r*row_stride : r*row_stride + vocab]):
 *   T = temperature[r] == 0  ->  argmax x (lowest index on ties).
 *   otherwise x' = x / T; keep the top_k[r] largest (exactly k, lowest index
 *   first among equal values; k <= 0 or k >= vocab keeps all); if top_p[r] < 1
 *   keep the smallest descending prefix of the kept set whose renormalised
 *   probability mass exceeds top_p[r], plus every id equal to its last value;
 *   token = argmax over kept j of x'_j + g_j, g_j = -log(-log u_j), with
 *   u_j = ((w_j >> 9) + 0.5) * 2^-23 and w_j word (j % 4) of Philox4x32-10
 *   (Salmon et al., SC'11) at key (lo32(seeds[r]), hi32(seeds[r])) and
 *   counter (j / 4, lo32(offsets[r]), hi32(offsets[r]), 0).
 * Inputs: logits (dtype) rows of `vocab` elements `row_stride` apart;
 *         temperature f32 [num_rows] (>= 0), top_k int32, top_p f32,
 *         seeds u64, offsets u64, all [num_rows] device arrays.
 * Output: token_ids int32 [num_rows].
 * Requirements: 1 <= vocab <= 2^23.  NaN logits give unspecified ids.
 */
pkvd_status pkvd_sample(int32_t* token_ids, const void* logits, int32_t dtype,
                        int32_t num_rows, int32_t vocab, int64_t row_stride,
                        const float* temperature, const int32_t* top_k, const float* top_p,
                        const uint64_t* seeds, const uint64_t* offsets,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * pkvd_sample_ex -- pkvd_sample plus the rest of Grok-1's sample_token
 * ("第 8 章 runners.py 推理引擎", section 8.3; TOP_K = 8 in section 8.3.2),
 * each part optional (NULL = off):
 *   mask      allowed-id bits [num_rows, mask_words_per_row] uint32, bit
 *             (j % 32) of word (j / 32) set = id j may be drawn.  A masked
 *             id counts as the page's logit -1e10 after the temperature: it
 *             is cut by every filter and never drawn while any id is allowed;
 *             a row with no allowed id draws uniformly over all ids (greedy
 *             rows take id 0).  Rows must be 16-byte aligned and short enough
 *             to sit in shared memory over a cluster (else
 *             PKVD_UNSUPPORTED_SHAPE).
 *   token_prob f32 [num_rows]: the drawn id's probability under softmax of
 *             the filtered logits (kept ids as scaled, all others 0); 1 for
 *             greedy rows.
 *   top_probs f32 [num_rows, 8], top_ids int32 [num_rows, 8]: the 8 largest
 *             of those probabilities -- kept ids by value, index order among
 *             equal values, then ids of probability 0 in index order (-1 and
 *             0 past the vocabulary).  Greedy rows: the drawn id with 1, then
 *             the lowest other ids with 0.
 * workspace: at least pkvd_sample_workspace_bytes(num_rows, vocab) bytes
 *             (4-byte aligned) when any of token_prob / top_probs / top_ids
 *             is requested (the sampler leaves each row's cut there for a
 *             second kernel); otherwise unused.
 * The token ids are those pkvd_sample gives for the same inputs.
 */
pkvd_status pkvd_sample_ex(int32_t* token_ids, const void* logits, int32_t dtype,
                           int32_t num_rows, int32_t vocab, int64_t row_stride,
                           const float* temperature, const int32_t* top_k, const float* top_p,
                           const uint64_t* seeds, const uint64_t* offsets,
                           const uint32_t* mask, int64_t mask_words_per_row,
                           float* token_prob, float* top_probs, int32_t* top_ids,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Host block manager -- the allocation side of the paged cache (nano-vllm
 * "Model Runner" notes, section "prepare Prefill": schedule-time CPU
 * bookkeeping that fills each sequence's block table and counts its
 * prefix-cached tokens; nanochat "04 · Engine 推理与工具调用", sections 2-3:
 * one prefill cloned N ways, here by sharing blocks).  Host memory and host
 * calls only; one object per cache, not thread-safe.
 *   - free blocks form a FIFO (0 .. num_blocks-1 at the start): allocation
 *     takes the front, a block whose reference count drops to 0 goes to the
 *     back and keeps its content key until it is handed out again;
 *   - a full block is keyed by (the block before it in the table, or -1, and
 *     its block_size token ids); a prompt reuses its registered full blocks
 *     in order up to the first miss, never the block holding its last token;
 *   - a token written into a shared last block first gets a fresh copy of it
 *     (copy-on-write: the caller copies the rows with pkvd_copy_blocks);
 *   - a request that needs more free blocks than there are returns
 *     PKVD_NO_SPACE and changes nothing.
 */
typedef struct pkvd_block_manager pkvd_block_manager;

pkvd_status pkvd_bm_create(int32_t num_blocks, int32_t block_size, pkvd_block_manager** out);
void pkvd_bm_destroy(pkvd_block_manager* bm);
/* Free blocks; -1 for a NULL manager. */
int32_t pkvd_bm_num_free(const pkvd_block_manager* bm);
/* Reference count of one block; -1 if out of range. */
int32_t pkvd_bm_ref_count(const pkvd_block_manager* bm, int32_t block);

/* A new prompt of num_tokens token ids (host array): writes its block table
 * (host, at most max_blocks entries), the block count and the number of
 * leading tokens already cached (a multiple of block_size). */
pkvd_status pkvd_bm_allocate(pkvd_block_manager* bm, const int32_t* tokens, int32_t num_tokens,
                             int32_t* block_table, int32_t max_blocks, int32_t* num_blocks,
                             int32_t* cached_tokens);

/* The sequence grew by one token: tokens holds all num_tokens ids, the table
 * the blocks of the first num_tokens - 1 (*num_blocks of them; updated in
 * place).  When the new token lands in a shared block, *copy_src / *copy_dst
 * / *copy_rows name the copy-on-write copy to run before the store (else
 * -1, -1, 0). */
pkvd_status pkvd_bm_append(pkvd_block_manager* bm, const int32_t* tokens, int32_t num_tokens,
                           int32_t* block_table, int32_t* num_blocks, int32_t max_blocks,
                           int32_t* copy_src, int32_t* copy_dst, int32_t* copy_rows);

/* A clone of a sequence: every block of the table gains a reference (the
 * caller keeps a copy of the table for the clone). */
pkvd_status pkvd_bm_fork(pkvd_block_manager* bm, const int32_t* block_table, int32_t num_blocks);

/* A sequence ends: every block of its table loses a reference (last first). */
pkvd_status pkvd_bm_release(pkvd_block_manager* bm, const int32_t* block_table, int32_t num_blocks);

/* The prefix a decode batch shares, for pkvd_paged_decode_attention_prefix:
 * the longest run of leading table entries that name the same physical
 * block in every row, counting only blocks that every row holds in full
 * before its newest token (so every context passes the prefix), in tokens
 * (a multiple of block_size; 0 for fewer than two rows).  block_tables and
 * context_lens are HOST arrays ([num_seqs][table_stride], [num_seqs]), as the
 * scheduler keeps them; nothing is read on the device. */
pkvd_status pkvd_bm_shared_prefix(const int32_t* block_tables, int32_t num_seqs, int32_t table_stride,
                                  const int32_t* context_lens, int32_t block_size, int32_t* prefix_tokens);

/*
 * pkvd_copy_blocks -- the device side of copy-on-write: for each i < count,
 * the first rows[i] token rows of block src[i] (K and V, every head) are
 * copied to block dst[i].  src, dst, rows: device int32 [count].
 * Device errors: a block id outside the pool or rows outside [0, block_size]
 * sets PKVD_ERR_BLOCK_ID and that copy is skipped.
 */
pkvd_status pkvd_copy_blocks(const pkvd_cache* cache, const int32_t* src, const int32_t* dst,
                             const int32_t* rows, int32_t count, void* stream, int32_t* err_flag);

#ifdef __cplusplus
}
#endif

#endif /* PKVD_H */
