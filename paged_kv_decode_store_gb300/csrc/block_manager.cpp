// Host block manager: physical KV-cache blocks for sequences, with exact
// prefix sharing, clone-N and copy-on-write of a shared partial block.
//
// nano-vllm "Model Runner" notes, section "prepare Prefill": block
// allocation is CPU-side bookkeeping done at schedule time; can_allocate
// consults the prefix cache, allocate writes physical block ids into the
// sequence's block table, num_cached_tokens counts the prompt tokens already
// in the cache.  nanochat "04 · Engine 推理与工具调用", sections 2-3: one
// prefill, then N clones of the cache -- here clones share blocks by
// reference count.
//
// Rules (the pages stop at the interface):
// * free blocks form a FIFO (0, 1, ..., n-1 at the start): allocation takes
//   the front, a block whose count drops to 0 goes to the back.  The FIFO is
//   an intrusive doubly linked list, so a cached free block can be reclaimed
//   from the middle in O(1).
// * a full block is keyed by (the block before it in the table, or -1, and
//   its block_size token ids) -- an exact key; a freed block keeps its key
//   until it is handed out again.
// * a prompt looks its full blocks up in order, stops at the first miss and
//   never looks up the block holding its last token.
// * a token written into a shared last block (count > 1) first gets a fresh
//   copy of it (the caller copies the rows with pkvd_copy_blocks); a block
//   that becomes full registers its key.
// * a request that needs more free blocks than there are changes nothing.
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "pkvd.h"

struct pkvd_block_manager {
  int32_t nb, bs;
  std::vector<int32_t> ref;
  std::vector<int32_t> prev, next;      // free FIFO links (-1 = none)
  std::vector<uint8_t> in_free;
  int32_t head = -1, tail = -1, nfree = 0;
  std::vector<std::string> key_of;      // empty: not registered
  std::unordered_map<std::string, int32_t> cache;

  pkvd_block_manager(int32_t n, int32_t b)
      : nb(n), bs(b), ref(n, 0), prev(n, -1), next(n, -1), in_free(n, 0), key_of(n) {
    for (int32_t i = 0; i < n; ++i) push_back(i);
  }
  void push_back(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b;
    else head = b;
    tail = b;
    in_free[b] = 1;
    ++nfree;
  }
  void unlink(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b];
    else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b];
    else tail = prev[b];
    prev[b] = next[b] = -1;
    in_free[b] = 0;
    --nfree;
  }
  std::string key(int32_t parent, const int32_t* tokens) const {
    std::string k(sizeof(int32_t) * (size_t)(bs + 1), '\0');
    std::memcpy(&k[0], &parent, sizeof(int32_t));
    std::memcpy(&k[sizeof(int32_t)], tokens, sizeof(int32_t) * (size_t)bs);
    return k;
  }
  int32_t take() {                      // the FIFO front, its stale key forgotten
    const int32_t b = head;
    unlink(b);
    if (!key_of[b].empty()) {
      cache.erase(key_of[b]);
      key_of[b].clear();
    }
    ref[b] = 1;
    return b;
  }
  void register_block(int32_t b, int32_t parent, const int32_t* tokens) {
    std::string k = key(parent, tokens);
    if (cache.count(k)) return;         // an equal block is registered: keep the first
    key_of[b] = k;
    cache.emplace(std::move(k), b);
  }
};

extern "C" {

pkvd_status pkvd_bm_create(int32_t num_blocks, int32_t block_size, pkvd_block_manager** out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PKVD_INVALID_ARG;
  *out = nullptr;
  pkvd_block_manager* bm = new (std::nothrow) pkvd_block_manager(num_blocks, block_size);
  if (!bm) return PKVD_NO_SPACE;
  *out = bm;
  return PKVD_OK;
}

void pkvd_bm_destroy(pkvd_block_manager* bm) { delete bm; }

int32_t pkvd_bm_num_free(const pkvd_block_manager* bm) { return bm ? bm->nfree : -1; }

int32_t pkvd_bm_ref_count(const pkvd_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->nb) return -1;
  return bm->ref[block];
}

pkvd_status pkvd_bm_allocate(pkvd_block_manager* bm, const int32_t* tokens, int32_t num_tokens,
                             int32_t* block_table, int32_t max_blocks, int32_t* num_blocks,
                             int32_t* cached_tokens) {
  if (!bm || num_tokens <= 0 || !tokens || !block_table || !num_blocks || !cached_tokens) return PKVD_INVALID_ARG;
  const int32_t bs = bm->bs;
  const int32_t nblk = (num_tokens + bs - 1) / bs;
  if (nblk > max_blocks) return PKVD_INVALID_ARG;
  // prefix lookups: full blocks with at least one prompt token after them
  std::vector<int32_t> hits;
  int32_t parent = -1;
  for (int32_t i = 0; i < nblk && (int64_t)(i + 1) * bs <= num_tokens - 1; ++i) {
    auto it = bm->cache.find(bm->key(parent, tokens + (int64_t)i * bs));
    if (it == bm->cache.end()) break;
    hits.push_back(it->second);
    parent = it->second;
  }
  int32_t need = nblk - (int32_t)hits.size();
  for (int32_t b : hits) need += bm->ref[b] == 0;
  if (need > bm->nfree) return PKVD_NO_SPACE;
  int32_t n = 0;
  for (int32_t b : hits) {
    if (bm->ref[b] == 0) bm->unlink(b);
    ++bm->ref[b];
    block_table[n++] = b;
  }
  parent = n ? block_table[n - 1] : -1;
  for (int32_t i = n; i < nblk; ++i) {
    const int32_t b = bm->take();
    if ((int64_t)(i + 1) * bs <= num_tokens) bm->register_block(b, parent, tokens + (int64_t)i * bs);
    block_table[n++] = b;
    parent = b;
  }
  *num_blocks = n;
  *cached_tokens = bs * (int32_t)hits.size();
  return PKVD_OK;
}

pkvd_status pkvd_bm_append(pkvd_block_manager* bm, const int32_t* tokens, int32_t num_tokens, int32_t* block_table,
                           int32_t* num_blocks, int32_t max_blocks, int32_t* copy_src, int32_t* copy_dst,
                           int32_t* copy_rows) {
  if (!bm || !tokens || !block_table || !num_blocks || !copy_src || !copy_dst || !copy_rows || num_tokens <= 0)
    return PKVD_INVALID_ARG;
  const int32_t bs = bm->bs;
  const int32_t p = num_tokens - 1;     // the new token's position
  int32_t n = *num_blocks;
  if (n != (p + bs - 1) / bs) return PKVD_INVALID_ARG;   // the table covers the tokens before p
  *copy_src = *copy_dst = -1;
  *copy_rows = 0;
  if (p % bs == 0) {                    // a new block
    if (n >= max_blocks) return PKVD_INVALID_ARG;
    if (bm->nfree == 0) return PKVD_NO_SPACE;
    block_table[n++] = bm->take();
    *num_blocks = n;
  } else {
    const int32_t last = block_table[n - 1];
    if (last < 0 || last >= bm->nb) return PKVD_INVALID_ARG;
    if (bm->ref[last] > 1) {            // shared: copy before writing
      if (bm->nfree == 0) return PKVD_NO_SPACE;
      const int32_t b = bm->take();
      --bm->ref[last];
      *copy_src = last;
      *copy_dst = b;
      *copy_rows = p % bs;
      block_table[n - 1] = b;
    }
  }
  if (p % bs == bs - 1) {               // the last block is now full
    const int32_t i = p / bs;
    bm->register_block(block_table[i], i > 0 ? block_table[i - 1] : -1, tokens + (int64_t)i * bs);
  }
  return PKVD_OK;
}

pkvd_status pkvd_bm_fork(pkvd_block_manager* bm, const int32_t* block_table, int32_t num_blocks) {
  if (!bm || num_blocks < 0 || (num_blocks > 0 && !block_table)) return PKVD_INVALID_ARG;
  for (int32_t i = 0; i < num_blocks; ++i)
    if (block_table[i] < 0 || block_table[i] >= bm->nb || bm->ref[block_table[i]] <= 0) return PKVD_INVALID_ARG;
  for (int32_t i = 0; i < num_blocks; ++i) ++bm->ref[block_table[i]];
  return PKVD_OK;
}

pkvd_status pkvd_bm_shared_prefix(const int32_t* block_tables, int32_t num_seqs, int32_t table_stride,
                                  const int32_t* context_lens, int32_t block_size, int32_t* prefix_tokens) {
  if (!prefix_tokens || num_seqs < 0 || block_size <= 0 || table_stride < 0) return PKVD_INVALID_ARG;
  *prefix_tokens = 0;
  if (num_seqs < 2) return PKVD_OK;
  if (!block_tables || !context_lens) return PKVD_INVALID_ARG;
  // whole blocks that every row holds before its newest token, and that are
  // the same physical block in every row
  int64_t limit = table_stride;
  for (int32_t i = 0; i < num_seqs; ++i) {
    if (context_lens[i] <= 0) return PKVD_OK;
    const int64_t full = (int64_t)(context_lens[i] - 1) / block_size;
    if (full < limit) limit = full;
  }
  int64_t shared = 0;
  for (; shared < limit; ++shared) {
    const int32_t b = block_tables[shared];
    if (b < 0) break;
    bool same = true;
    for (int32_t i = 1; i < num_seqs && same; ++i) same = block_tables[(int64_t)i * table_stride + shared] == b;
    if (!same) break;
  }
  *prefix_tokens = (int32_t)(shared * block_size);
  return PKVD_OK;
}

pkvd_status pkvd_bm_release(pkvd_block_manager* bm, const int32_t* block_table, int32_t num_blocks) {
  if (!bm || num_blocks < 0 || (num_blocks > 0 && !block_table)) return PKVD_INVALID_ARG;
  for (int32_t i = 0; i < num_blocks; ++i)
    if (block_table[i] < 0 || block_table[i] >= bm->nb || bm->ref[block_table[i]] <= 0) return PKVD_INVALID_ARG;
  for (int32_t i = num_blocks - 1; i >= 0; --i) {
    const int32_t b = block_table[i];
    if (--bm->ref[b] == 0) bm->push_back(b);
  }
  return PKVD_OK;
}

}  // extern "C"
