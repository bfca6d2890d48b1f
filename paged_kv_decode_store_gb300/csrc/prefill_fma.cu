// Varlen paged prefill attention on the CUDA cores, for every cache dtype
// (the only prefill path for fp32 caches; the tensor-core paths need 16-bit
// K/V).  Same operation as prefill.cu and prefill_tc.cu (nano-vllm "Model
// Runner" notes, sections "prefix cache" and "prefill and decode": new token j
// of sequence i sits at position (k_len_i - q_len_i) + j and attends causally
// to positions 0..p of its sequence through the block table).
//
// One CTA per (new token row, KV head); warp w computes query head
// hk * G + w.  K and V rows are staged 32 keys at a time in shared memory as
// fp32 (padded rows: lane j reads key j without bank conflicts); lane j scores
// key j, the warp keeps an online softmax in the log2 domain and each lane
// accumulates D / 32 output dimensions.  Keys outside [ws(p), p] and rows of
// bad blocks are staged as zeros and masked.  Written for coverage, not speed.
#include "common.cuh"
#include "launch.h"

namespace pkvd {

namespace {

constexpr int kFmaKeys = 32;
constexpr int kFmaMaxGroup = 16;      // query heads per KV head (warps per CTA)

struct FmaParams {
  void* out;
  const void* q;
  const uint8_t* kc;
  const uint8_t* vc;
  int64_t num_blocks;
  int block_size;
  int64_t block_stride, token_stride, head_stride;   // elements
  const int32_t* tables;
  int max_blocks;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int num_seqs;
  int total_q;
  int hq;
  int group;
  float scale_log2;
  int window;
  int32_t* err;
};

__device__ __forceinline__ float fma_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T, int D>
__global__ void __launch_bounds__(32 * kFmaMaxGroup) prefill_fma_kernel(const FmaParams p) {
  __shared__ float ks[kFmaKeys][D + 1];
  __shared__ float vs[kFmaKeys][D + 1];
  __shared__ float qs[kFmaMaxGroup][D];
  const int t = blockIdx.x, hk = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;

  pdl_wait();
  pdl_trigger();

  if (t >= p.cu_q[p.num_seqs]) return;                    // a row past the batch: not written
  int lo = 0, hi = p.num_seqs - 1;                         // the last i with cu_q[i] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu_q[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int seq = lo;
  const int q0 = p.cu_q[seq], q1 = p.cu_q[seq + 1];
  const int klen = p.cu_k[seq + 1] - p.cu_k[seq], qlen = q1 - q0;
  if (t < q0 || t >= q1 || qlen < 0 || klen < qlen || q1 > p.total_q ||
      (int64_t)klen > (int64_t)p.max_blocks * p.block_size) {
    if (threadIdx.x == 0) flag_error(p.err, PKVD_ERR_CONTEXT);
    return;
  }
  const int pos = klen - qlen + (t - q0);
  const int ws = (p.window > 0 && pos + 1 > p.window) ? pos + 1 - p.window : 0;
  const int h = hk * G + warp;
  const T* q = static_cast<const T*>(p.q) + ((int64_t)t * p.hq + h) * D;
  for (int d = lane; d < D; d += 32) qs[warp][d] = DT<T>::to_f(q[d]);
  const int32_t* table = p.tables + (int64_t)seq * p.max_blocks;
  const T* kc = reinterpret_cast<const T*>(p.kc);
  const T* vc = reinterpret_cast<const T*>(p.vc);

  float m = -INFINITY, l = 0.f, o[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) o[i] = 0.f;
  for (int kbase = (ws / kFmaKeys) * kFmaKeys; kbase <= pos; kbase += kFmaKeys) {
    __syncthreads();                                       // the previous chunk is no longer read
    for (int e = threadIdx.x; e < kFmaKeys * D; e += blockDim.x) {
      const int r = e / D, d = e - (e / D) * D;
      const int kp = kbase + r;
      float kv = 0.f, vv = 0.f;
      if (kp >= ws && kp <= pos) {
        const int phys = table[kp / p.block_size];
        if (phys >= 0 && phys < p.num_blocks) {
          const int64_t off = (int64_t)phys * p.block_stride + (int64_t)(kp % p.block_size) * p.token_stride +
                              (int64_t)hk * p.head_stride + d;
          kv = DT<T>::to_f(kc[off]);
          vv = DT<T>::to_f(vc[off]);
        } else if (d == 0) {
          flag_error(p.err, PKVD_ERR_BLOCK_ID);            // the row reads as zeros
        }
      }
      ks[r][d] = kv;
      vs[r][d] = vv;
    }
    __syncthreads();
    // lane j scores key kbase + j
    const int kp = kbase + lane;
    float sc = -INFINITY;
    if (kp >= ws && kp <= pos) {
      float acc = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) acc = fmaf(qs[warp][d], ks[lane][d], acc);
      sc = acc * p.scale_log2;
    }
    float mx = sc;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, s));
    const float mn = fmaxf(m, mx);
    const float mu = mn == -INFINITY ? 0.f : mn;
    const float alpha = fma_ex2(m - mu);                   // 0 while nothing was seen yet
    const float pj = fma_ex2(sc - mu);
    float ps = pj;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) ps += __shfl_xor_sync(FULL_MASK, ps, s);
    l = l * alpha + ps;
    m = mn;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) o[i] *= alpha;
    for (int j = 0; j < kFmaKeys; ++j) {
      const float pjj = __shfl_sync(FULL_MASK, pj, j);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) o[i] = fmaf(pjj, vs[j][lane + 32 * i], o[i]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  T* out = static_cast<T*>(p.out) + ((int64_t)t * p.hq + h) * D;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) out[lane + 32 * i] = DT<T>::from_f(o[i] * inv);
}

template <typename T, int D>
cudaError_t launch_fma_typed(const FmaParams& prm, dim3 grid, int threads, cudaStream_t stream) {
  return launch_pdl(prefill_fma_kernel<T, D>, grid, dim3(threads), 0, stream, prm);
}

}  // namespace

bool prefill_fma_supported(int dtype, int head_dim, int group, int num_kv_heads) {
  return (dtype == PKVD_F32 || dtype == PKVD_F16 || dtype == PKVD_BF16) && (head_dim == 64 || head_dim == 128) &&
         group >= 1 && group <= kFmaMaxGroup && num_kv_heads <= 65535;
}

cudaError_t launch_prefill_fma(const PrefillArgs& a, cudaStream_t stream) {
  const pkvd_cache& c = a.cache;
  FmaParams prm;
  prm.out = a.out;
  prm.q = a.q;
  prm.kc = static_cast<const uint8_t*>(c.k_base);
  prm.vc = static_cast<const uint8_t*>(c.v_base);
  prm.num_blocks = c.num_blocks;
  prm.block_size = c.block_size;
  prm.block_stride = c.block_stride;
  prm.token_stride = c.token_stride;
  prm.head_stride = c.head_stride;
  prm.tables = a.block_tables;
  prm.max_blocks = a.max_blocks_per_seq;
  prm.cu_q = a.cu_seqlens_q;
  prm.cu_k = a.cu_seqlens_k;
  prm.num_seqs = a.num_seqs;
  prm.total_q = a.total_q;
  prm.hq = a.num_q_heads;
  prm.group = a.num_q_heads / c.num_kv_heads;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.window = a.window;
  prm.err = a.err;
  const dim3 grid(a.total_q, c.num_kv_heads);
  const int threads = 32 * prm.group;
  if (c.dtype == PKVD_F32)
    return c.head_dim == 64 ? launch_fma_typed<float, 64>(prm, grid, threads, stream)
                            : launch_fma_typed<float, 128>(prm, grid, threads, stream);
  if (c.dtype == PKVD_BF16)
    return c.head_dim == 64 ? launch_fma_typed<__nv_bfloat16, 64>(prm, grid, threads, stream)
                            : launch_fma_typed<__nv_bfloat16, 128>(prm, grid, threads, stream);
  return c.head_dim == 64 ? launch_fma_typed<__half, 64>(prm, grid, threads, stream)
                          : launch_fma_typed<__half, 128>(prm, grid, threads, stream);
}

}  // namespace pkvd
