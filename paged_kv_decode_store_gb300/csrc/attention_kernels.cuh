// Paged single-query GQA decode attention: partition kernel + LSE merge.
//
// What is computed (nano-vllm "Model Runner" notes, sections "prefill and
// decode" and "allocated kv cache"; Grok-1 "第 8 章 runners.py 推理引擎",
// sections 8.2.3 and 8.5): for row i, query head h, kv head hk = h / G,
//   out[i,h] = sum_{j < ctx_i} softmax_j(scale * <q[i,h], K_j>) V_j
// with K_j / V_j the row j % bs of physical block block_table[i][j / bs].
//
// GB300 design (the pages give no kernel; this one is HBM-bound by design):
// * Work = the flattened list of (sequence, 16-token chunk) pairs over all
//   rows.  A persistent grid of one CTA per SM takes an equal contiguous
//   slice of that list (stream-K style), so every SM moves the same number
//   of K/V bytes whatever the length mix.  A slice may start or end inside
//   a sequence; such partial segments leave an unnormalised (m, l, acc)
//   record in the workspace and the merge kernel, launched as a
//   programmatic dependent so its launch overlaps this kernel's tail,
//   combines them with the log-sum-exp identity.  Segments wholly inside one
//   CTA are normalised and written directly.
// * One producer warp walks the slice, looks block ids up (32 table entries
//   per coalesced load, shuffled to the lane that needs them) and issues
//   cp.async.bulk (TMA engine) copies of each chunk's K and V token rows --
//   all KV heads of a row are contiguous in the cache -- into a ring of
//   shared-memory stages, completion counted on an mbarrier.  Smem rows are
//   padded by 16 bytes so that 8 consecutive token rows of one head fall in
//   8 different bank groups (conflict-free ldmatrix).
// * Eight consumer warps each own KV head(s); every query head of a GQA
//   group is computed from the one staged K/V read.  Two consumer variants:
//   - FMA: fp32 dot products, 16-byte smem vectors, xor-shuffle reductions,
//     fp32 online softmax in the log2 domain.
//   - MMA (16-bit caches): S^T[16 tok x 8 heads] = K_tile Q^T with
//     mma.m16n8k16 (the GQA group is the N=8 dimension, no waste for G=8),
//     online softmax on the accumulator fragment, P^T re-used as the B
//     operand after a movmatrix transpose, O^T += V^T P^T with ldmatrix.trans.
// * Rows past a context and stale smem rows are removed with selects, never
//   by multiplying with 0 (the cache may hold NaN there); for the tensor-core
//   path the stale V rows of a partial chunk are zeroed first.
// * Every wait is bounded (mbar_wait_bounded): a broken pipeline sets
//   PKVD_ERR_TIMEOUT and the CTA leaves after draining its own copies.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace pkvd {

enum : int { F_FIRST = 1, F_LAST = 2, F_COMPLETE = 4, F_SLOT1 = 8 };

struct PartParams {
  void* out;
  const void* q;
  const uint8_t* k_base;
  const uint8_t* v_base;
  int64_t block_stride, token_stride, head_stride;   // elements
  int64_t num_blocks;
  int block_size, hkv, hq, G;
  const int32_t* tables;
  int max_blocks;
  const int32_t* ctx;
  int ctx_cap;
  int window;          // > 0: attend to the newest `window` positions only
  int num_seqs;
  float scale_log2;
  float* rec;          // partial records [grid][2][hq][D + 4]: acc[D], m, l, pad (the workspace)
  int32_t* err;
  int stages;
  int rowb;            // padded smem bytes of one token row (all heads)
  int row_bytes;       // hkv * D * sizeof(T)
  int rows_contig;     // heads of a token row adjacent in memory
  int active_warps;    // consumer warps that own heads
};

// The partition kernel's parameters for a call (attention.cu); `rec` is the
// record area of the workspace.
PartParams part_params(const AttnArgs& a, float* rec);

// First attended position of a context of c tokens: the newest `window`
// positions with a sliding window (window > 0), else 0.
__device__ __forceinline__ int window_start(int c, int window) { return (window > 0 && c > window) ? c - window : 0; }

// 16-token chunks of row i's attended span (length clamped to [0, cap]).
__device__ __forceinline__ int chunks_of(const int32_t* ctx, int i, int cap, int window) {
  int c = ctx[i];
  c = c < 0 ? 0 : (c > cap ? cap : c);
  return (c - window_start(c, window) + kChunk - 1) / kChunk;
}

__device__ __forceinline__ int64_t slice_begin(int64_t C, int cta, int grid) {
  return (C * cta) / grid;
}

// Block-wide inclusive scan of one int per thread (blockDim = kAttnThreads).
__device__ __forceinline__ int block_incl_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kAttnThreads / 32;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(FULL_MASK, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  int base = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int t = s_warp[w];
    if (w < warp) base += t;
    total += t;
  }
  __syncthreads();
  return v + base;
}

struct SmemHdr {
  uint64_t full[4];
  uint64_t empty[4];
  int4 meta[4];
  int scan_warp[kAttnThreads / 32];
  int found_seq;
  int found_off;
  long long total;
  int abort_flag;
};

// ----------------------------------------------------------- consumers
template <typename T, int D, int HPW, int GMAX>
struct FmaConsumer {
  static constexpr int ESZ = sizeof(T);
  static constexpr int VEC = 16 / ESZ;
  static constexpr int LPT = D * ESZ / 16;   // lanes per token row of one head
  static constexpr int TPP = 32 / LPT;       // tokens per warp pass
  static_assert(LPT >= 1 && LPT <= 32, "head row must be 16..512 bytes");

  float q[HPW][GMAX][VEC];
  float acc[HPW][GMAX][VEC];
  float m[HPW][GMAX], l[HPW][GMAX];

  __device__ void begin(const PartParams& p, int seq, int warp, int lane) {
    const int li = lane % LPT;
    const T* qb = static_cast<const T*>(p.q);
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const int hk = warp * HPW + j;
#pragma unroll
      for (int g = 0; g < GMAX; ++g) {
        float f[VEC];
        if (g < p.G) {
          const uint4 u = *reinterpret_cast<const uint4*>(
              qb + ((int64_t)seq * p.hq + hk * p.G + g) * D + li * VEC);
          Vec16<T>::unpack(u, f);
        } else {
#pragma unroll
          for (int v = 0; v < VEC; ++v) f[v] = 0.f;
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          q[j][g][v] = f[v] * p.scale_log2;
          acc[j][g][v] = 0.f;
        }
        m[j][g] = -INFINITY;
        l[j][g] = 0.f;
      }
    }
  }

  __device__ void chunk(const PartParams& p, const uint8_t* sK, const uint8_t* sV, int ntok,
                        int warp, int lane) {
    const int grp = lane / LPT, li = lane % LPT;
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const int hk = warp * HPW + j;
      const int col = hk * D * ESZ + li * 16;
#pragma unroll 2
      for (int t0 = 0; t0 < kChunk; t0 += TPP) {
        const int t = t0 + grp;
        const bool valid = t < ntok;
        float kf[VEC];
        Vec16<T>::unpack(*reinterpret_cast<const uint4*>(sK + t * p.rowb + col), kf);
        float s[GMAX];
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
          float d = 0.f;
#pragma unroll
          for (int v = 0; v < VEC; ++v) d = fmaf(q[j][g][v], kf[v], d);
#pragma unroll
          for (int o = LPT / 2; o > 0; o >>= 1) d += __shfl_xor_sync(FULL_MASK, d, o);
          s[g] = d;
        }
        if (valid) {
          float vf[VEC];
          Vec16<T>::unpack(*reinterpret_cast<const uint4*>(sV + t * p.rowb + col), vf);
#pragma unroll
          for (int g = 0; g < GMAX; ++g) {
            if (g < p.G) {
              const float mn = fmaxf(m[j][g], s[g]);
              const float corr = exp2f(m[j][g] - mn);
              const float pr = exp2f(s[g] - mn);
              l[j][g] = l[j][g] * corr + pr;
#pragma unroll
              for (int v = 0; v < VEC; ++v) acc[j][g][v] = fmaf(acc[j][g][v], corr, pr * vf[v]);
              m[j][g] = mn;
            }
          }
        }
      }
    }
  }

  __device__ void finish(const PartParams& p, int seq, int flags, int cta, int warp, int lane, long long P,
                         long long nrow, long long C, int grid) {
    const int li = lane % LPT;
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const int hk = warp * HPW + j;
#pragma unroll
      for (int g = 0; g < GMAX; ++g) {
        // combine the TPP independent token-group states of the warp
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) {
          const float mo = __shfl_xor_sync(FULL_MASK, m[j][g], o);
          const float lo = __shfl_xor_sync(FULL_MASK, l[j][g], o);
          const float mn = fmaxf(m[j][g], mo);
          const float ca = (m[j][g] == -INFINITY) ? 0.f : exp2f(m[j][g] - mn);
          const float cb = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const float ao = __shfl_xor_sync(FULL_MASK, acc[j][g][v], o);
            acc[j][g][v] = acc[j][g][v] * ca + ao * cb;
          }
          l[j][g] = l[j][g] * ca + lo * cb;
          m[j][g] = mn;
        }
        if (g < p.G && lane < LPT) {
          const int h = hk * p.G + g;
          if (flags & F_COMPLETE) {
            const float inv = 1.f / l[j][g];
            T* o = static_cast<T*>(p.out) + ((int64_t)seq * p.hq + h) * D + li * VEC;
            alignas(16) T tmp[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) tmp[v] = DT<T>::from_f(acc[j][g][v] * inv);
            *reinterpret_cast<uint4*>(o) = *reinterpret_cast<const uint4*>(tmp);
          } else {
            const int slot = (flags & F_SLOT1) ? 1 : 0;
            float* r = p.rec + ((int64_t)(cta * 2 + slot) * p.hq + h) * (D + 4);
#pragma unroll
            for (int v = 0; v < VEC; ++v) r[li * VEC + v] = acc[j][g][v];
            if (li == 0) {
              r[D] = m[j][g];
              r[D + 1] = l[j][g];
            }
          }
        }
      }
    }
  }
};

template <typename T, int D, int HPW>
struct MmaConsumer {
  static constexpr int ESZ = sizeof(T);
  static constexpr int KS = D / 16;     // k-steps of QK^T, m-tiles of V^T P^T
  static_assert(ESZ == 2, "tensor-core path is for 16-bit caches");

  uint32_t qf[HPW][KS][2];
  float acc[HPW][KS][4];
  float m[HPW][2], l[HPW][2];

  __device__ void begin(const PartParams& p, int seq, int warp, int lane) {
    const int lr = lane >> 2, lc = lane & 3;
    const T* qb = static_cast<const T*>(p.q);
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const int hk = warp * HPW + j;
      const T* row = qb + ((int64_t)seq * p.hq + hk * p.G + lr) * D;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qf[j][kk][0] = lr < p.G ? *reinterpret_cast<const uint32_t*>(row + kk * 16 + 2 * lc) : 0u;
        qf[j][kk][1] = lr < p.G ? *reinterpret_cast<const uint32_t*>(row + kk * 16 + 8 + 2 * lc) : 0u;
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[j][kk][r] = 0.f;
      }
      m[j][0] = m[j][1] = -INFINITY;
      l[j][0] = l[j][1] = 0.f;
    }
  }

  __device__ void chunk(const PartParams& p, uint8_t* sK, uint8_t* sV, int ntok, int warp, int lane) {
    const int lr = lane >> 2;
    // ldmatrix row/column providers: A = K tile (row-major, rows = tokens)
    const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int a_col = (lane >> 4) * 16;                       // bytes
    // A = V^T via .trans: source rows = tokens, 8 dims each
    const int v_mat = lane >> 3;
    const int v_row = (lane & 7) + (v_mat >> 1) * 8;
    const int v_col = (v_mat & 1) * 8 * ESZ;                  // bytes
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const int hk = warp * HPW + j;
      const int hoff = hk * D * ESZ;
      if (ntok < kChunk) {
        // stale rows of a partial chunk: zero this head's V slice so that
        // P = 0 never meets a NaN in the tensor-core product
        constexpr int VPR = D * ESZ / 16;
        for (int idx = lane; idx < (kChunk - ntok) * VPR; idx += 32) {
          const int r = ntok + idx / VPR, c = idx % VPR;
          *reinterpret_cast<uint4*>(sV + r * p.rowb + hoff + c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t kaddr = smem_u32(sK) + a_row * p.rowb + hoff + a_col;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t a[4];
        ldsm_x4(kaddr + kk * 32, a[0], a[1], a[2], a[3]);
        Mma<T>::run(s, a, qf[j][kk][0], qf[j][kk][1]);
      }
      // fragment: s0,s1 -> token lr, heads 2lc,2lc+1 ; s2,s3 -> token lr+8
      const float sl = p.scale_log2;
      const float x0 = lr < ntok ? s[0] * sl : -INFINITY;
      const float x1 = lr < ntok ? s[1] * sl : -INFINITY;
      const float x2 = lr + 8 < ntok ? s[2] * sl : -INFINITY;
      const float x3 = lr + 8 < ntok ? s[3] * sl : -INFINITY;
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, o));
      }
      const float mn0 = fmaxf(m[j][0], mx0), mn1 = fmaxf(m[j][1], mx1);
      const float c0 = exp2f(m[j][0] - mn0), c1 = exp2f(m[j][1] - mn1);
      const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
      const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
      l[j][0] = l[j][0] * c0 + p0 + p2;
      l[j][1] = l[j][1] * c1 + p1 + p3;
      m[j][0] = mn0;
      m[j][1] = mn1;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        acc[j][mt][0] *= c0;
        acc[j][mt][1] *= c1;
        acc[j][mt][2] *= c0;
        acc[j][mt][3] *= c1;
      }
      const uint32_t b0 = movmatrix_trans(Mma<T>::pack(p0, p1));
      const uint32_t b1 = movmatrix_trans(Mma<T>::pack(p2, p3));
      const uint32_t vaddr = smem_u32(sV) + v_row * p.rowb + hoff + v_col;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(vaddr + mt * 16 * ESZ, a[0], a[1], a[2], a[3]);
        Mma<T>::run(acc[j][mt], a, b0, b1);
      }
    }
  }

  __device__ void finish(const PartParams& p, int seq, int flags, int cta, int warp, int lane, long long P,
                         long long nrow, long long C, int grid) {
    const int lr = lane >> 2, lc = lane & 3;
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const int hk = warp * HPW + j;
      float lA = l[j][0], lB = l[j][1];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        lA += __shfl_xor_sync(FULL_MASK, lA, o);
        lB += __shfl_xor_sync(FULL_MASK, lB, o);
      }
      const int gA = 2 * lc, gB = 2 * lc + 1;
      if (flags & F_COMPLETE) {
        const float iA = 1.f / lA, iB = 1.f / lB;
        T* ob = static_cast<T*>(p.out) + ((int64_t)seq * p.hq + hk * p.G) * D;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d0 = mt * 16 + lr;
          if (gA < p.G) {
            ob[gA * D + d0] = DT<T>::from_f(acc[j][mt][0] * iA);
            ob[gA * D + d0 + 8] = DT<T>::from_f(acc[j][mt][2] * iA);
          }
          if (gB < p.G) {
            ob[gB * D + d0] = DT<T>::from_f(acc[j][mt][1] * iB);
            ob[gB * D + d0 + 8] = DT<T>::from_f(acc[j][mt][3] * iB);
          }
        }
      } else {
        const int slot = (flags & F_SLOT1) ? 1 : 0;
        float* rb = p.rec + ((int64_t)(cta * 2 + slot) * p.hq + hk * p.G) * (D + 4);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d0 = mt * 16 + lr;
          if (gA < p.G) {
            rb[gA * (D + 4) + d0] = acc[j][mt][0];
            rb[gA * (D + 4) + d0 + 8] = acc[j][mt][2];
          }
          if (gB < p.G) {
            rb[gB * (D + 4) + d0] = acc[j][mt][1];
            rb[gB * (D + 4) + d0 + 8] = acc[j][mt][3];
          }
        }
        if (lr == 0) {
          if (gA < p.G) { rb[gA * (D + 4) + D] = m[j][0]; rb[gA * (D + 4) + D + 1] = lA; }
          if (gB < p.G) { rb[gB * (D + 4) + D] = m[j][1]; rb[gB * (D + 4) + D + 1] = lB; }
        }
      }
    }
  }
};

// ------------------------------------------------------ partition kernel
template <typename T, int D, typename Consumer>
__global__ void __launch_bounds__(kAttnThreads, 1) paged_decode_partition_kernel(const PartParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemHdr& hdr = *reinterpret_cast<SmemHdr*>(smem_raw);
  uint8_t* stage_base = smem_raw + ((sizeof(SmemHdr) + 127) / 128) * 128;
  const int stage_bytes = 2 * kChunk * p.rowb;
  const int S = p.stages;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, grid = gridDim.x;
  // Everything up to the producer's first copy reads only inputs of this call
  // (context lengths, block tables, q), never memory the previous kernel (the
  // KV store) writes, so it runs before the dependency wait and overlaps that
  // kernel; the producer waits before its first cache read.

  // ---- scan the chunk counts: total, this CTA's slice, and its first row
  // (every CTA computes the same scan; CTA 0 flags bad lengths)
  if (tid == 0) {
    hdr.found_seq = -1;
    hdr.found_off = 0;
    hdr.abort_flag = 0;
  }
  long long C, c0, c1;
  if (p.num_seqs <= kAttnThreads) {
    // one row per thread: a single block scan gives the total and the row offsets
    const int i = tid;
    const int n = i < p.num_seqs ? chunks_of(p.ctx, i, p.ctx_cap, p.window) : 0;
    if (cta == 0 && i < p.num_seqs) {
      const int raw = p.ctx[i];
      if (raw < 0 || raw > p.ctx_cap) flag_error(p.err, PKVD_ERR_CONTEXT);
    }
    int total;
    const int incl = block_incl_scan(n, hdr.scan_warp, total);   // also orders the header writes
    C = total;
    c0 = slice_begin(C, cta, grid);
    c1 = slice_begin(C, cta + 1, grid);
    if (c0 >= c1 && cta != 0) return;
    const int excl = incl - n;
    if (n > 0 && excl <= c0 && c0 < excl + n) {
      hdr.found_seq = i;
      hdr.found_off = (int)(c0 - excl);
    }
    __syncthreads();
  } else {
    long long part = 0;
    for (int i = tid; i < p.num_seqs; i += kAttnThreads) part += chunks_of(p.ctx, i, p.ctx_cap, p.window);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL_MASK, part, o);
    if (tid == 0) hdr.total = 0;
    __syncthreads();
    if (lane == 0) atomicAdd(reinterpret_cast<unsigned long long*>(&hdr.total), (unsigned long long)part);
    __syncthreads();
    C = hdr.total;
    c0 = slice_begin(C, cta, grid);
    c1 = slice_begin(C, cta + 1, grid);
    if (c0 >= c1 && cta != 0) return;
    int running = 0;
    for (int base = 0; base < p.num_seqs; base += kAttnThreads) {
      const int i = base + tid;
      const int n = i < p.num_seqs ? chunks_of(p.ctx, i, p.ctx_cap, p.window) : 0;
      int total;
      const int incl = block_incl_scan(n, hdr.scan_warp, total);
      const int excl = running + incl - n;
      if (cta == 0 && i < p.num_seqs) {
        const int raw = p.ctx[i];
        if (raw < 0 || raw > p.ctx_cap) flag_error(p.err, PKVD_ERR_CONTEXT);
      }
      if (i < p.num_seqs && n > 0 && excl <= c0 && c0 < excl + n) {
        hdr.found_seq = i;
        hdr.found_off = (int)(c0 - excl);
      }
      running += total;
      __syncthreads();
      if (cta != 0 && hdr.found_seq >= 0) break;
    }
  }
  // the merge kernel may be scheduled now; it waits for this grid to finish
  if (tid == 0) pdl_trigger();
  if (c0 >= c1) return;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hdr.full[s], 1);
      mbar_init(&hdr.empty[s], p.active_warps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int nit = (int)(c1 - c0);
  const int esz = sizeof(T);

  if (warp == kConsumerWarps) {
    // =============================== producer warp
    int seq = hdr.found_seq, ch = hdr.found_off;
    int ctx_seq = min(max(p.ctx[seq], 0), p.ctx_cap);
    int tok_base = window_start(ctx_seq, p.window);
    int nch = (ctx_seq - tok_base + kChunk - 1) / kChunk;
    int seg_start = ch;
    long long row_start = c0 - ch;          // flat index of the row's chunk 0
    bool first_seg = true;
    int tb_seq = -1, tb_base = 0, tb_val = -1;
    if (nch > 0) {            // the first table window, fetched before the wait
      const int lb = (tok_base + ch * kChunk) / p.block_size;
      tb_seq = seq;
      tb_base = lb;
      tb_val = lb + lane < p.max_blocks ? p.tables[(int64_t)seq * p.max_blocks + lb + lane] : -1;
    }
    pdl_wait();               // the cache rows stored by the previous kernel
    int it = 0;
    for (; it < nit; ++it) {
      while (ch >= nch && seq + 1 < p.num_seqs) {
        row_start += nch;
        ++seq;
        ctx_seq = min(max(p.ctx[seq], 0), p.ctx_cap);
        tok_base = window_start(ctx_seq, p.window);
        nch = (ctx_seq - tok_base + kChunk - 1) / kChunk;
        ch = 0;
        seg_start = 0;
        first_seg = false;
      }
      if (ch >= nch) break;     // unreachable: the slice never passes the last chunk
      const int stage = it % S;
      const int n = it / S;
      if (n > 0 && !mbar_wait_bounded(&hdr.empty[stage], (n - 1) & 1)) {
        if (lane == 0) { flag_error(p.err, PKVD_ERR_TIMEOUT); hdr.abort_flag = 1; }
        break;
      }
      if (*reinterpret_cast<volatile int*>(&hdr.abort_flag)) break;
      const int token0 = tok_base + ch * kChunk;
      const int ntok = min(kChunk, ctx_seq - token0);
      // a chunk of 16 consecutive positions spans at most two blocks (it
      // starts on a 16-token boundary unless a sliding window moved it)
      const int lb0 = token0 / p.block_size, off0 = token0 % p.block_size;
      const int lb1 = (token0 + max(ntok, 1) - 1) / p.block_size;
      if (seq != tb_seq || lb0 < tb_base || lb1 >= tb_base + 32) {
        tb_seq = seq;
        tb_base = lb0;
        const int e = lb0 + lane;
        tb_val = e < p.max_blocks ? p.tables[(int64_t)seq * p.max_blocks + e] : -1;
      }
      const int phys0 = __shfl_sync(FULL_MASK, tb_val, lb0 - tb_base);
      const int phys1 = __shfl_sync(FULL_MASK, tb_val, lb1 - tb_base);
      const bool ok = phys0 >= 0 && phys0 < p.num_blocks && phys1 >= 0 && phys1 < p.num_blocks;
      const int ncopy = ok ? ntok : 0;
      int flags = 0;
      if (ch == seg_start) flags |= F_FIRST;
      if (ch == nch - 1 || it == nit - 1) flags |= F_LAST;
      if (seg_start == 0 && (c0 + it - ch + nch - 1) < c1) flags |= F_COMPLETE;
      if (!first_seg) flags |= F_SLOT1;
      if (lane == 0) {
        if (!ok) flag_error(p.err, PKVD_ERR_BLOCK_ID);
        hdr.meta[stage] = make_int4(seq, ncopy, flags | (nch << 4), (int)row_start);
        mbar_arrive_expect_tx(&hdr.full[stage], (uint32_t)(ncopy * 2 * p.row_bytes));
      }
      __syncwarp();
      if (ncopy > 0) {
        uint8_t* sdst = stage_base + stage * stage_bytes;
        // row t of the chunk: block phys0 row off0 + t before the block
        // boundary, block phys1 row off0 + t - block_size after it
        const int split = p.block_size - off0;
        const int64_t b0 = ((int64_t)phys0 * p.block_stride + (int64_t)off0 * p.token_stride) * esz;
        const int64_t b1 = ((int64_t)phys1 * p.block_stride - (int64_t)split * p.token_stride) * esz;
        if (p.rows_contig) {
          for (int r = lane; r < 2 * ncopy; r += 32) {
            const int kv = r >= ncopy;
            const int t = kv ? r - ncopy : r;
            const int64_t src = (t < split ? b0 : b1) + (int64_t)t * p.token_stride * esz;
            bulk_g2s(sdst + kv * kChunk * p.rowb + t * p.rowb, (kv ? p.v_base : p.k_base) + src, p.row_bytes,
                     &hdr.full[stage]);
          }
        } else {
          const int per = ncopy * p.hkv;
          for (int r = lane; r < 2 * per; r += 32) {
            const int kv = r >= per;
            const int rem = kv ? r - per : r;
            const int t = rem / p.hkv, h = rem % p.hkv;
            const int64_t src = (t < split ? b0 : b1) + ((int64_t)t * p.token_stride + (int64_t)h * p.head_stride) * esz;
            bulk_g2s(sdst + kv * kChunk * p.rowb + t * p.rowb + h * D * esz, (kv ? p.v_base : p.k_base) + src,
                     D * esz, &hdr.full[stage]);
          }
        }
      }
      ++ch;
    }
    // drain: every copy this warp issued has landed before the CTA leaves
    const int first = it > S ? it - S : 0;
    for (int k = first; k < it; ++k) {
      if (!mbar_wait_bounded(&hdr.full[k % S], (k / S) & 1)) {
        if (lane == 0) flag_error(p.err, PKVD_ERR_TIMEOUT);
        break;
      }
    }
    return;
  }

  // ================================== consumer warps
  if (warp >= p.active_warps) return;
  Consumer cons;
  for (int it = 0; it < nit; ++it) {
    const int stage = it % S;
    if (!mbar_wait_bounded(&hdr.full[stage], (it / S) & 1)) {
      if (lane == 0) { flag_error(p.err, PKVD_ERR_TIMEOUT); hdr.abort_flag = 1; }
      break;
    }
    const int4 meta = hdr.meta[stage];
    const int seq = meta.x, ntok = meta.y, flags = meta.z & 15;
    const int nrow = meta.z >> 4;
    const long long row_start = meta.w;
    if (flags & F_FIRST) cons.begin(p, seq, warp, lane);
    uint8_t* sK = stage_base + stage * stage_bytes;
    uint8_t* sV = sK + kChunk * p.rowb;
    if (ntok > 0) cons.chunk(p, sK, sV, ntok, warp, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&hdr.empty[stage]);
    if (flags & F_LAST) cons.finish(p, seq, flags, cta, warp, lane, row_start, nrow, C, grid);
  }
}

// ------------------------------------------------------------ merge
// One CTA per row and group of 256 output float4 slices (blockIdx.y), so
// rows with many heads spread over several SMs; launched as a programmatic
// dependent of the partition kernel: it waits for that grid, then combines the partial records of the
// CTAs whose slices cut the row (log-sum-exp identity), writes zeros for an
// empty context, and leaves rows one CTA finished on its own untouched.
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  o = sum_s 2^(m_s - M) acc_s / L
// Each thread owns float4 output slices; for every chunk of 8 records all
// loads are issued before any is used (one L2 round trip per chunk).
constexpr int kMaxMergeRecords = 1024;     // >= any partition grid (one CTA per SM)

template <typename T>
__global__ void __launch_bounds__(256) lse_merge_kernel(T* __restrict__ out, const float* __restrict__ rec,
                                                        const int32_t* __restrict__ ctx, int ctx_cap, int window,
                                                        int num_seqs, int hq, int D, int grid, int parts) {
  __shared__ int s_rec[kMaxMergeRecords];
  __shared__ int s_n;
  __shared__ long long s_part[2][8];
  const int i = blockIdx.x;
  // Row i's chunk range [P, P + n) and the total C from the context lengths.
  // They are read before pdl_wait(), so this part overlaps the partition
  // kernel -- and possibly the kernel before it, since the partition kernel
  // lets this grid start before its own dependency wait.  That is safe by the
  // input contract of the attention call: context_lens is written by no
  // kernel that lets its dependents start early (the library's own kernels
  // never write it).  The partial records are read after pdl_wait().
  long long before = 0, all = 0;
  for (int r = threadIdx.x; r < num_seqs; r += blockDim.x) {
    const int c = chunks_of(ctx, r, ctx_cap, window);
    all += c;
    if (r < i) before += c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(FULL_MASK, before, o);
    all += __shfl_xor_sync(FULL_MASK, all, o);
  }
  if ((threadIdx.x & 31) == 0) {
    s_part[0][threadIdx.x >> 5] = before;
    s_part[1][threadIdx.x >> 5] = all;
  }
  __syncthreads();
  long long P = 0, C = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    P += s_part[0][w];
    C += s_part[1][w];
  }
  const long long n = chunks_of(ctx, i, ctx_cap, window);
  T* orow = out + (int64_t)i * hq * D;
  if (n <= 0) {
    pdl_wait();
    pdl_trigger();
    for (int idx = blockIdx.y * blockDim.x + threadIdx.x; idx < hq * D; idx += gridDim.y * blockDim.x)
      orow[idx] = DT<T>::from_f(0.f);
    return;
  }
  const int a = (int)(((P + 1) * grid - 1) / C);
  const int b = (int)(((P + n) * grid - 1) / C);
  if (a == b) {                     // written by one CTA on its own
    pdl_wait();
    pdl_trigger();
    return;
  }
  if (threadIdx.x == 0) {
    // CTA a's slice starts at or before P (its record of this row is its
    // last segment unless it starts exactly at P); later CTAs start inside
    // the row.  Empty slices (only when C < grid) are skipped.
    const bool a_at_start = (C * a) / grid == P;
    int cnt = 0;
    for (int c = a; c <= b && cnt < kMaxMergeRecords; ++c) {
      if (C < grid && (C * c) / grid >= (C * (c + 1)) / grid) continue;
      s_rec[cnt++] = c * 2 + ((c == a && !a_at_start) ? 1 : 0);
    }
    s_n = cnt;
  }
  __syncthreads();
  const int nrec = s_n;
  pdl_wait();                       // the partition kernel's records
  pdl_trigger();
  // `parts` adjacent lanes (1, 2 or 4) share one float4 output slice: part
  // p takes records p, p + parts, ..., so a row cut into many pieces needs
  // fewer rounds of record loads; the parts' states are then combined with
  // shuffles (the same identity).
  const int Q = D / 4;
  constexpr int R = 8;
  const int nslots = hq * Q * parts;
  for (int base = blockIdx.y * blockDim.x; base < nslots; base += gridDim.y * blockDim.x) {
    const int t = base + threadIdx.x;                 // whole warps iterate together
    const int sl = t / parts, part = t % parts;
    const bool live = t < nslots;
    const int h = live ? sl / Q : 0, d4 = live ? (sl % Q) * 4 : 0;
    float M = -INFINITY, L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = part; live && k0 < nrec; k0 += R * parts) {
      float mk[R], lk[R];
      float4 ak[R];
#pragma unroll
      for (int e = 0; e < R; ++e) {
        const int k = k0 + e * parts;
        mk[e] = -INFINITY;
        lk[e] = 0.f;
        ak[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < nrec) {
          const float* r = rec + ((int64_t)s_rec[k] * hq + h) * (D + 4);
          mk[e] = r[D];
          lk[e] = r[D + 1];
          ak[e] = *reinterpret_cast<const float4*>(r + d4);
        }
      }
#pragma unroll
      for (int e = 0; e < R; ++e) {
        const float m = mk[e];
        if (m == -INFINITY) continue;
        const float Mn = fmaxf(M, m);
        const float cs = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
        const float cr = exp2f(m - Mn);
        L = L * cs + lk[e] * cr;
        o.x = o.x * cs + ak[e].x * cr;
        o.y = o.y * cs + ak[e].y * cr;
        o.z = o.z * cs + ak[e].z * cr;
        o.w = o.w * cs + ak[e].w * cr;
        M = Mn;
      }
    }
    for (int off = 1; off < parts; off <<= 1) {      // lanes of one slice are adjacent
      const float Mo = __shfl_xor_sync(FULL_MASK, M, off);
      const float Lo = __shfl_xor_sync(FULL_MASK, L, off);
      const float ox = __shfl_xor_sync(FULL_MASK, o.x, off), oy = __shfl_xor_sync(FULL_MASK, o.y, off);
      const float oz = __shfl_xor_sync(FULL_MASK, o.z, off), ow = __shfl_xor_sync(FULL_MASK, o.w, off);
      const float Mn = fmaxf(M, Mo);
      const float ca = M == -INFINITY ? 0.f : exp2f(M - Mn);
      const float cb = Mo == -INFINITY ? 0.f : exp2f(Mo - Mn);
      L = L * ca + Lo * cb;
      o.x = o.x * ca + ox * cb;
      o.y = o.y * ca + oy * cb;
      o.z = o.z * ca + oz * cb;
      o.w = o.w * ca + ow * cb;
      M = Mn;
    }
    if (live && part == 0) {
      const float inv = 1.f / L;
      T* dst = orow + h * D + d4;
      dst[0] = DT<T>::from_f(o.x * inv);
      dst[1] = DT<T>::from_f(o.y * inv);
      dst[2] = DT<T>::from_f(o.z * inv);
      dst[3] = DT<T>::from_f(o.w * inv);
    }
  }
}

// -------------------------------------------------------- launch helper
inline size_t smem_header_bytes() { return ((sizeof(SmemHdr) + 127) / 128) * 128; }

// The dynamic shared-memory limit is a per-device property of the kernel, so
// it is set on every launch (a host-side call, no stream work): a process that
// drives several GPUs, or several threads, needs no shared bookkeeping.
template <typename T, int D, typename Consumer>
cudaError_t launch_partition(const PartParams& pp, int grid, size_t smem, cudaStream_t stream) {
  auto kern = paged_decode_partition_kernel<T, D, Consumer>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kAttnThreads), smem, stream, pp);
}

}  // namespace pkvd
