// Decode-attention launch: grid sizing, workspace layout, path choice, and
// the merge kernel that follows the partition kernel.
#include "attention_dispatch.cuh"

namespace pkvd {

namespace {
constexpr int kMaxDynSmem = 232448;    // 227 KB opt-in per CTA on sm_100-family parts

int elem_bytes(int dtype) { return dtype == PKVD_F32 ? 4 : 2; }

int stage_count(int dtype, int head_dim, int num_kv_heads) {
  const size_t rowb = (size_t)num_kv_heads * head_dim * elem_bytes(dtype) + 16;
  const size_t stage = 2 * kChunk * rowb;
  const size_t avail = kMaxDynSmem - smem_header_bytes();
  const size_t s = avail / stage;
  return s > 4 ? 4 : (int)s;
}

int group_bound(int g) { return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8; }
}  // namespace

int attention_grid(int num_seqs, int max_context_len, int sm_count) {
  if (num_seqs <= 0 || max_context_len <= 0 || sm_count <= 0) return 0;
  const long long units = (long long)num_seqs * ((max_context_len + kChunk - 1) / kChunk);
  long long g = units < sm_count ? units : sm_count;
  return (int)(g < kMaxMergeRecords ? g : kMaxMergeRecords);
}

size_t attention_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int grid) {
  (void)num_seqs;
  return (size_t)grid * 2 * num_q_heads * (head_dim + 4) * sizeof(float);
}

bool attention_path_supported(int path, int dtype, int head_dim, int num_kv_heads, int group) {
  if (head_dim != 64 && head_dim != 128) return false;
  if (group < 1 || group > 8) return false;
  if (!(num_kv_heads >= 1 && (num_kv_heads <= 8 || num_kv_heads == 16))) return false;
  if (stage_count(dtype, head_dim, num_kv_heads) < 2) return false;
  if (path == PKVD_PATH_MMA) return dtype != PKVD_F32 && (num_kv_heads == 8 || num_kv_heads == 16);
  if (path == PKVD_PATH_FMA) return dtype != PKVD_F32 || num_kv_heads <= 8;
  return false;
}

int attention_default_path(int dtype, int head_dim, int num_kv_heads, int group) {
  if (attention_path_supported(PKVD_PATH_MMA, dtype, head_dim, num_kv_heads, group)) return PKVD_PATH_MMA;
  if (attention_path_supported(PKVD_PATH_FMA, dtype, head_dim, num_kv_heads, group)) return PKVD_PATH_FMA;
  return 0;
}

PartParams part_params(const AttnArgs& a, float* rec) {
  const int esz = elem_bytes(a.dtype);
  PartParams pp;
  pp.out = a.out;
  pp.q = a.q;
  pp.k_base = static_cast<const uint8_t*>(a.k_base);
  pp.v_base = static_cast<const uint8_t*>(a.v_base);
  pp.block_stride = a.block_stride;
  pp.token_stride = a.token_stride;
  pp.head_stride = a.head_stride;
  pp.num_blocks = a.num_blocks;
  pp.block_size = a.block_size;
  pp.hkv = a.num_kv_heads;
  pp.hq = a.num_q_heads;
  pp.G = a.num_q_heads / a.num_kv_heads;
  pp.tables = a.block_tables;
  pp.max_blocks = a.max_blocks_per_seq;
  pp.ctx = a.context_lens;
  const long long cap = (long long)a.max_blocks_per_seq * a.block_size;
  pp.ctx_cap = (int)(cap < a.max_context_len ? cap : a.max_context_len);
  pp.window = a.window;
  pp.num_seqs = a.num_seqs;
  pp.scale_log2 = a.scale * 1.4426950408889634f;
  pp.rec = rec;
  pp.err = a.err;
  pp.stages = stage_count(a.dtype, a.head_dim, a.num_kv_heads);
  pp.row_bytes = a.num_kv_heads * a.head_dim * esz;
  pp.rowb = pp.row_bytes + 16;
  pp.rows_contig = a.head_stride == a.head_dim ? 1 : 0;
  pp.active_warps = a.num_kv_heads == 16 ? kConsumerWarps : a.num_kv_heads;
  return pp;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  const int esz = elem_bytes(a.dtype);
  const int G = a.num_q_heads / a.num_kv_heads;
  float* rec = static_cast<float*>(a.workspace);
  if (a.grid > 0) {
    PartParams pp = part_params(a, rec);    const int hpw = a.num_kv_heads == 16 ? 2 : 1;
    pp.active_warps = hpw == 2 ? kConsumerWarps : a.num_kv_heads;
    const size_t smem = smem_header_bytes() + (size_t)pp.stages * 2 * kChunk * pp.rowb;
    const int gmax = group_bound(G);
    cudaError_t e;
    if (a.dtype == PKVD_F32) e = partition_f32(pp, a.head_dim, hpw, gmax, a.path, a.grid, smem, stream);
    else if (a.dtype == PKVD_F16) e = partition_f16(pp, a.head_dim, hpw, gmax, a.path, a.grid, smem, stream);
    else e = partition_bf16(pp, a.head_dim, hpw, gmax, a.path, a.grid, smem, stream);
    if (e != cudaSuccess) return e;
  }
  if (a.num_seqs == 0) return cudaSuccess;
  if (a.grid == 0) {
    // no context anywhere: every output row is zero
    return cudaMemsetAsync(a.out, 0, (size_t)a.num_seqs * a.num_q_heads * a.head_dim * esz, stream);
  }
  // the merge kernel as a programmatic dependent of the partition kernel
  const long long cap_all = (long long)a.max_blocks_per_seq * a.block_size;
  const int ctx_cap = (int)(cap_all < a.max_context_len ? cap_all : a.max_context_len);
  // lanes per output slice: enough that a row's records load in one round of
  // eight per lane (rows are cut into about grid / num_seqs + 1 pieces)
  const int pieces = a.grid / a.num_seqs + 1;
  const int parts = pieces > 16 ? 4 : pieces > 8 ? 2 : 1;
  const int groups = (a.num_q_heads * (a.head_dim / 4) * parts + 255) / 256;
  const dim3 mg((unsigned)a.num_seqs, (unsigned)groups), mb(256);
  if (a.dtype == PKVD_F32)
    return launch_pdl(lse_merge_kernel<float>, mg, mb, 0, stream, static_cast<float*>(a.out), (const float*)rec,
                      a.context_lens, ctx_cap, a.window, a.num_seqs, a.num_q_heads, a.head_dim, a.grid, parts);
  if (a.dtype == PKVD_F16)
    return launch_pdl(lse_merge_kernel<__half>, mg, mb, 0, stream, static_cast<__half*>(a.out), (const float*)rec,
                      a.context_lens, ctx_cap, a.window, a.num_seqs, a.num_q_heads, a.head_dim, a.grid, parts);
  return launch_pdl(lse_merge_kernel<__nv_bfloat16>, mg, mb, 0, stream, static_cast<__nv_bfloat16*>(a.out),
                    (const float*)rec, a.context_lens, ctx_cap, a.window, a.num_seqs, a.num_q_heads, a.head_dim, a.grid, parts);
}

}  // namespace pkvd
