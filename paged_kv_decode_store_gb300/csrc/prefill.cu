// Varlen paged prefill attention: every newly scheduled token of every
// sequence attends causally to its sequence's cached prefix and to the new
// tokens up to itself, all read through the block table from the paged cache
// (after this step's store).
//
// nano-vllm "Model Runner" notes, section "prefix cache": the batch is given
// by cu_seqlens_q (tokens scheduled now) and cu_seqlens_k (scheduled plus
// cached), so sequence i's new token j sits at position
// (k_len_i - q_len_i) + j; section "prefill and decode": prefill is the
// dense, compute-bound phase and gets its own kernel, separate from the
// memory-bound decode kernel.
//
// Design (sm_103a, 16-bit K/V):
// * One CTA per (KV head, sequence, tile of query tokens).  The G query heads
//   that share the KV head are packed into the tile's 128 M rows
//   (row = token * G + head-in-group), so every K/V tile loaded from the
//   cache serves the whole group.  Tiles are counted from the end of each
//   sequence and the tile index is the slowest grid dimension: the heaviest
//   tiles (most keys under the causal mask) of every sequence start first.
// * 8 warps, 16 rows each.  Q stays in registers as m16n8k16 A fragments;
//   per 64-key tile, S = Q K^T and O += P V run on the tensor cores
//   (mma.sync, fp32 accumulation) with an online softmax in between
//   (base-2 exponent, running max and sum per row, P rounded to the input
//   type for the second product).
// * K/V tiles are gathered row by row (the block table resolves each key's
//   physical block) with 16-byte cp.async into padded shared-memory rows
//   (row pitch D + 8 elements: conflict-free ldmatrix), double buffered so
//   the next tile streams in while the current one is multiplied.  Keys
//   outside [first window start of the tile, last position of the tile]
//   are zero-filled, never read.
// * The causal / window mask is only evaluated on tiles that cross a row's
//   diagonal or window edge; a warp skips tiles none of its rows can see.
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace pkvd {

namespace {

constexpr int kPfThreads = 256;
constexpr int kPfRows = 128;   // M rows per CTA (8 warps x 16)
constexpr int kPfKeys = 64;    // keys per K/V tile

template <int D>
struct PfLayout {
  static constexpr int kPitch = D + 8;                       // elements per shared row
  static constexpr int kQBytes = kPfRows * kPitch * 2;
  static constexpr int kTileBytes = kPfKeys * kPitch * 2;    // K or V of one tile
  static constexpr int kBytes = kQBytes + 4 * kTileBytes;    // Q + 2 stages of (K, V)
  static constexpr int kChunks = D * 2 / 16;                 // 16-byte pieces per row
};

struct PfParams {
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
  int total_q;
  int hq;
  int group;
  int tile_tokens;     // query tokens per CTA (kPfRows / group)
  float scale_log2;    // softmax scale * log2(e)
  int window;
  int32_t* err;
};

__device__ __forceinline__ int pf_window_start(int c, int window) {
  return (window > 0 && c > window) ? c - window : 0;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_attention_kernel(const PfParams p) {
  using L = PfLayout<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int hk = blockIdx.x, seq = blockIdx.y, ztile = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();      // the cache rows of this step come from the store kernel
  pdl_trigger();

  const int q0 = p.cu_q[seq], q1 = p.cu_q[seq + 1];
  const int klen = p.cu_k[seq + 1] - p.cu_k[seq];
  const int qlen = q1 - q0;
  if (q0 < 0 || qlen < 0 || klen < qlen || q1 > p.total_q ||
      (int64_t)klen > (int64_t)p.max_blocks * p.block_size) {
    if (threadIdx.x == 0 && ztile == 0 && hk == 0) flag_error(p.err, PKVD_ERR_CONTEXT);
    return;
  }
  if (ztile == 0 && hk == 0 && threadIdx.x == 0 && qlen > (int)gridDim.z * p.tile_tokens)
    flag_error(p.err, PKVD_ERR_CONTEXT);   // longer than max_seqlen_q: the earliest tokens are not computed
  const int tok_end = qlen - ztile * p.tile_tokens;
  if (tok_end <= 0) return;
  const int tok_begin = max(0, tok_end - p.tile_tokens);
  const int G = p.group;
  const int qrows = (tok_end - tok_begin) * G;
  const int cached = klen - qlen;
  const int pos_first = cached + tok_begin, pos_last = cached + tok_end - 1;
  const int lo = pf_window_start(pos_first + 1, p.window);    // first key any row reads
  const int hi = pos_last;                                      // last key any row reads
  const int kt_first = lo / kPfKeys, kt_last = hi / kPfKeys;

  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + L::kQBytes;   // stage s: K at sKV + 2s*tile, V right after

  // ---- Q tile: row r = token * G + head-in-group; padding rows zero-filled
  {
    const T* q = static_cast<const T*>(p.q);
    for (int idx = threadIdx.x; idx < kPfRows * L::kChunks; idx += kPfThreads) {
      const int r = idx / L::kChunks, c = idx % L::kChunks;
      const bool ok = r < qrows;
      const int tt = r / G, g = r - tt * G;
      const int64_t row = ok ? ((int64_t)(q0 + tok_begin + tt) * p.hq + (int64_t)hk * G + g) : 0;
      cp_async16(sQ + (r * L::kPitch + c * 8) * 2, q + row * D + c * 8, ok);
    }
  }

  // ---- K/V tile kt into stage st (rows outside [lo, hi] zero-filled)
  const int32_t* table = p.tables + (int64_t)seq * p.max_blocks;
  auto load_kv = [&](int kt, int st) {
    const int kbase = kt * kPfKeys;
    const uint32_t dk = sKV + st * 2 * L::kTileBytes, dv = dk + L::kTileBytes;
    for (int idx = threadIdx.x; idx < kPfKeys * L::kChunks; idx += kPfThreads) {
      const int r = idx / L::kChunks, c = idx % L::kChunks;
      const int kp = kbase + r;
      bool ok = kp >= lo && kp <= hi;
      int64_t off = 0;
      if (ok) {
        const int phys = __ldg(table + kp / p.block_size);
        if (phys < 0 || phys >= p.num_blocks) {
          ok = false;
          if (c == 0) flag_error(p.err, PKVD_ERR_BLOCK_ID);
        } else {
          off = (int64_t)phys * p.block_stride + (int64_t)(kp % p.block_size) * p.token_stride +
                (int64_t)hk * p.head_stride + c * 8;
        }
      }
      const uint32_t d = (r * L::kPitch + c * 8) * 2;
      cp_async16(dk + d, p.kc + off * 2, ok);
      cp_async16(dv + d, p.vc + off * 2, ok);
    }
  };

  load_kv(kt_first, 0);
  cp_async_commit();

  // ---- per-warp and per-thread row bookkeeping
  const int row0 = warp * 16;
  const bool warp_live = row0 < qrows;
  const int wlast = min(row0 + 15, qrows - 1);
  const int w_pos_min = pos_first + row0 / G, w_pos_max = pos_first + wlast / G;
  const int w_ws_min = pf_window_start(w_pos_min + 1, p.window);
  const int w_ws_max = pf_window_start(w_pos_max + 1, p.window);
  const int ra = row0 + (lane >> 2), rb = ra + 8;
  const int pa = pos_first + ra / G, pb = pos_first + rb / G;
  const int wsa = pf_window_start(pa + 1, p.window), wsb = pf_window_start(pb + 1, p.window);

  uint32_t qf[D / 16][4];
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int kt = kt_first; kt <= kt_last; ++kt) {
    const int st = (kt - kt_first) & 1;
    if (kt < kt_last) {
      load_kv(kt + 1, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    if (kt == kt_first && warp_live) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(sQ + (r * L::kPitch + c) * 2, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }

    const int kbase = kt * kPfKeys;
    // A warp works on a tile only if one of its rows can see one of its keys.
    if (warp_live && kbase <= w_pos_max && kbase + kPfKeys - 1 >= w_ws_min) {
      const uint32_t sK = sKV + st * 2 * L::kTileBytes, sV = sK + L::kTileBytes;
      float s[kPfKeys / 8][4];
#pragma unroll
      for (int n = 0; n < kPfKeys / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < kPfKeys / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          const int r = np * 16 + (lane >> 4) * 8 + (lane & 7);
          const int c = kk * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(sK + (r * L::kPitch + c) * 2, b0, b1, b2, b3);
          Mma<T>::run(s[2 * np], qf[kk], b0, b1);
          Mma<T>::run(s[2 * np + 1], qf[kk], b2, b3);
        }
      }
      const bool masked = kbase + kPfKeys - 1 > w_pos_min || kbase < w_ws_max;
#pragma unroll
      for (int n = 0; n < kPfKeys / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = s[n][e] * p.scale_log2;
          if (masked) {
            const int kp = kbase + n * 8 + 2 * (lane & 3) + (e & 1);
            const int pr = e < 2 ? pa : pb, wr = e < 2 ? wsa : wsb;
            if (kp > pr || kp < wr) x = -INFINITY;
          }
          s[n][e] = x;
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < kPfKeys / 8; ++n) {
        mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
        mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
      const float a0 = ex2(m0 - u0), a1 = ex2(m1 - u1);
      m0 = n0;
      m1 = n1;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int n = 0; n < kPfKeys / 8; ++n) {
        s[n][0] = ex2(s[n][0] - u0);
        s[n][1] = ex2(s[n][1] - u0);
        s[n][2] = ex2(s[n][2] - u1);
        s[n][3] = ex2(s[n][3] - u1);
        rs0 += s[n][0] + s[n][1];
        rs1 += s[n][2] + s[n][3];
      }
      l0 = l0 * a0 + rs0;
      l1 = l1 * a1 + rs1;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= a0;
        o[i][1] *= a0;
        o[i][2] *= a1;
        o[i][3] *= a1;
      }
#pragma unroll
      for (int kk = 0; kk < kPfKeys / 16; ++kk) {
        uint32_t a[4];
        a[0] = Mma<T>::pack(s[2 * kk][0], s[2 * kk][1]);
        a[1] = Mma<T>::pack(s[2 * kk][2], s[2 * kk][3]);
        a[2] = Mma<T>::pack(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = Mma<T>::pack(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t b0, b1, b2, b3;
          const int r = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
          const int c = dp * 16 + (lane >> 4) * 8;
          ldsm_x4_trans(sV + (r * L::kPitch + c) * 2, b0, b1, b2, b3);
          Mma<T>::run(o[2 * dp], a, b0, b1);
          Mma<T>::run(o[2 * dp + 1], a, b2, b3);
        }
      }
    }
    __syncthreads();   // the stage is refilled by the next iteration's prefetch
  }

  if (!warp_live) return;
  l0 += __shfl_xor_sync(FULL_MASK, l0, 1);
  l0 += __shfl_xor_sync(FULL_MASK, l0, 2);
  l1 += __shfl_xor_sync(FULL_MASK, l1, 1);
  l1 += __shfl_xor_sync(FULL_MASK, l1, 2);
  const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
  T* out = static_cast<T*>(p.out);
  const int col = 2 * (lane & 3);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rb : ra;
    if (r >= qrows) continue;
    const int tt = r / G, g = r - tt * G;
    T* dst = out + ((int64_t)(q0 + tok_begin + tt) * p.hq + (int64_t)hk * G + g) * D + col;
    const float inv = half ? i1 : i0;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const uint32_t w = Mma<T>::pack(o[i][2 * half] * inv, o[i][2 * half + 1] * inv);
      *reinterpret_cast<uint32_t*>(dst + i * 8) = w;
    }
  }
}

template <typename T, int D>
cudaError_t launch_prefill_typed(const PfParams& prm, dim3 grid, cudaStream_t stream) {
  constexpr int smem = PfLayout<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(prefill_attention_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(prefill_attention_kernel<T, D>, grid, dim3(kPfThreads), smem, stream, prm);
}

}  // namespace

bool prefill_supported(int dtype, int head_dim, int group) {
  return (dtype == PKVD_F16 || dtype == PKVD_BF16) && (head_dim == 64 || head_dim == 128) && group >= 1 &&
         group <= kPfRows;
}

int prefill_tile_tokens(int group) { return kPfRows / group; }

cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream) {
  const int G = a.num_q_heads / a.cache.num_kv_heads;
  PfParams prm;
  prm.out = a.out;
  prm.q = a.q;
  prm.kc = static_cast<const uint8_t*>(a.cache.k_base);
  prm.vc = static_cast<const uint8_t*>(a.cache.v_base);
  prm.num_blocks = a.cache.num_blocks;
  prm.block_size = a.cache.block_size;
  prm.block_stride = a.cache.block_stride;
  prm.token_stride = a.cache.token_stride;
  prm.head_stride = a.cache.head_stride;
  prm.tables = a.block_tables;
  prm.max_blocks = a.max_blocks_per_seq;
  prm.cu_q = a.cu_seqlens_q;
  prm.cu_k = a.cu_seqlens_k;
  prm.total_q = a.total_q;
  prm.hq = a.num_q_heads;
  prm.group = G;
  prm.tile_tokens = prefill_tile_tokens(G);
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.window = a.window;
  prm.err = a.err;
  const int tiles = (a.max_seqlen_q + prm.tile_tokens - 1) / prm.tile_tokens;
  const dim3 grid(a.cache.num_kv_heads, a.num_seqs, tiles);
  const int D = a.cache.head_dim;
  if (a.cache.dtype == PKVD_BF16)
    return D == 64 ? launch_prefill_typed<__nv_bfloat16, 64>(prm, grid, stream)
                   : launch_prefill_typed<__nv_bfloat16, 128>(prm, grid, stream);
  return D == 64 ? launch_prefill_typed<__half, 64>(prm, grid, stream)
                 : launch_prefill_typed<__half, 128>(prm, grid, stream);
}

}  // namespace pkvd
