// Fused decode sampler: temperature, top-k, nucleus cut, Gumbel-max draw.
//
// Semantics (Grok-1 "第 8 章 runners.py 推理引擎", sections 8.3 sample_token
// and 8.3.1 top_p_filter; nanochat "04 · Engine" section 3 top-k; nano-vllm
// "Model Runner" notes, "run model": Gumbel-max sampler):
//   T <= 0 : argmax, lowest index on ties.
//   else   : x' = x / T; keep the k largest (exactly k; lowest index first
//            among equal values); keep the smallest descending prefix of
//            that set whose renormalised mass exceeds p, widened to every id
//            equal to its last value; token = argmax_kept x'_j + g_j with
//            Gumbel noise from Philox4x32-10 (Salmon et al., SC'11).
//
// No sort.  One CTA (1024 threads) per row, a few streaming passes over the
// row (L2-resident after the first):
//   1. max key and its lowest index (greedy result, softmax shift m).
//   2. top-k: MSB-first radix select, 8 bits per pass, on order-preserving
//      integer keys of the raw logits (16-bit keys for fp16/bf16, 32-bit for
//      fp32) -- exact, so the top-k set matches bit for bit.
//   3. nucleus: the same radix select, but each bin accumulates probability
//      mass exp((x - m)/T) in 2^-40 fixed point (64-bit integer atomics, so
//      the sums are exact and independent of thread order).  It finds the
//      key tau where the descending cumulative mass first exceeds p * Z.
//   4. Gumbel pass over the kept ids.  Only ids with x'_j >= max x' - 21 can
//      win (u is in [2^-24, 1 - 2^-24], so g lies in [-2.81, 16.64]); the
//      others are skipped exactly, which leaves a handful of Philox
//      evaluations for peaked rows.
// Ties at the k-th key are resolved by index (a radix select over the tie
// group's indices), only when the tie group straddles the cut.
#include "common.cuh"
#include "launch.h"

namespace pkvd {

constexpr int kSampThreads = 1024;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kHistCopies = 16;
constexpr float kGumbelSpan = 21.0f;

template <typename T> struct Keys;
template <> struct Keys<float> {
  static constexpr int BITS = 32;
  __device__ static uint32_t bits(float x) { return __float_as_uint(x); }
  __device__ static uint32_t key(uint32_t u) {
    if ((u & 0x7fffffffu) == 0) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  __device__ static float value(uint32_t u) { return __uint_as_float(u); }
  __device__ static float value_of_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
  }
};
template <> struct Keys<__half> {
  static constexpr int BITS = 16;
  __device__ static uint32_t key(uint32_t b) {
    if ((b & 0x7fffu) == 0) b = 0;
    return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
  }
  __device__ static float value(uint32_t b) {
    const unsigned short s = (unsigned short)b;
    return __half2float(*reinterpret_cast<const __half*>(&s));
  }
  __device__ static float value_of_key(uint32_t k) {
    return value((k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu));
  }
};
template <> struct Keys<__nv_bfloat16> {
  static constexpr int BITS = 16;
  __device__ static uint32_t key(uint32_t b) { return Keys<__half>::key(b); }
  __device__ static float value(uint32_t b) { return __uint_as_float(b << 16); }
  __device__ static float value_of_key(uint32_t k) {
    return value((k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu));
  }
};

// Order-preserving key of an fp32 score (for the argmax packing).
__device__ __forceinline__ uint32_t f32_order_key(float x) { return Keys<float>::key(__float_as_uint(x)); }

// Visit every element of a row: f(index, raw bits).  Vector loads of 16 bytes
// when the row is aligned; four loads in flight per thread.
template <typename T, typename F>
__device__ __forceinline__ void for_each_elem(const T* row, int V, bool vec_ok, F&& f) {
  constexpr int E = 16 / sizeof(T);
  if (vec_ok) {
    const int nv = V / E;
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    int v = threadIdx.x;
    for (; v + 3 * kSampThreads < nv; v += 4 * kSampThreads) {
      uint4 u[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) u[r] = __ldg(rv + v + r * kSampThreads);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t w[4] = {u[r].x, u[r].y, u[r].z, u[r].w};
        const int j0 = (v + r * kSampThreads) * E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint32_t b = (sizeof(T) == 4) ? w[e] : ((w[e / 2] >> (16 * (e & 1))) & 0xffffu);
          f(j0 + e, b);
        }
      }
    }
    for (; v < nv; v += kSampThreads) {
      const uint4 u = __ldg(rv + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint32_t b = (sizeof(T) == 4) ? w[e] : ((w[e / 2] >> (16 * (e & 1))) & 0xffffu);
        f(v * E + e, b);
      }
    }
    for (int j = nv * E + threadIdx.x; j < V; j += kSampThreads) {
      f(j, sizeof(T) == 4 ? __float_as_uint(*reinterpret_cast<const float*>(row + j))
                          : (uint32_t)(*reinterpret_cast<const unsigned short*>(row + j)));
    }
  } else {
    for (int j = threadIdx.x; j < V; j += kSampThreads) {
      f(j, sizeof(T) == 4 ? __float_as_uint(*reinterpret_cast<const float*>(row + j))
                          : (uint32_t)(*reinterpret_cast<const unsigned short*>(row + j)));
    }
  }
}

__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(FULL_MASK, v, o);
    v = t > v ? t : v;
  }
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  v = s[0];
  for (int w = 1; w < kSampWarps; ++w) v = s[w] > v ? s[w] : v;
  return v;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
    const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    if (r < 9) {
      k.x += W0;
      k.y += W1;
    }
  }
  return c;
}

__device__ __forceinline__ float gumbel_noise(uint64_t seed, uint64_t offset, uint32_t j) {
  const uint4 ctr = make_uint4(j >> 2, (uint32_t)offset, (uint32_t)(offset >> 32), 0u);
  const uint4 w4 = philox4x32_10(ctr, make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
  const uint32_t sel = j & 3u;
  const uint32_t w = sel == 0 ? w4.x : (sel == 1 ? w4.y : (sel == 2 ? w4.z : w4.w));
  const float u = (__uint2float_rn(w >> 9) + 0.5f) * 1.1920928955078125e-07f;   // * 2^-23, exact
  return -logf(-logf(u));
}

struct SampSmem {
  unsigned long long hist[kHistCopies][256];   // counts (low 32 bits used) or fixed-point mass
  unsigned long long tot[256];
  unsigned long long red[kSampWarps];
  int sel_bin;
  unsigned long long sel_before;
  int found;
};

// Clear the private histograms.
__device__ __forceinline__ void hist_clear(SampSmem& sm) {
  unsigned long long* h = &sm.hist[0][0];
  for (int i = threadIdx.x; i < kHistCopies * 256; i += kSampThreads) h[i] = 0ull;
}

// Sum the private copies into tot[].
__device__ __forceinline__ void hist_total(SampSmem& sm) {
  if (threadIdx.x < 256) {
    unsigned long long s = 0;
#pragma unroll
    for (int c = 0; c < kHistCopies; ++c) s += sm.hist[c][threadIdx.x];
    sm.tot[threadIdx.x] = s;
  }
}

// Warp 0 scans tot[] from bin 255 down and finds the first bin where
// before + tot[b] crosses the target: for counts the condition is
// before + tot[b] >= target (target = remaining k), for mass it is
// before + tot[b] > target.  Writes sel_bin (-1 if none) and sel_before.
__device__ __forceinline__ void select_bin(SampSmem& sm, unsigned long long target, bool strict) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  unsigned long long v[8], local = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    v[e] = sm.tot[255 - (lane * 8 + e)];
    local += v[e];
  }
  unsigned long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
  }
  unsigned long long before = incl - local;
  int found = -1;
  unsigned long long fb = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const unsigned long long after = before + v[e];
    const bool hit = strict ? (after > target) : (after >= target);
    if (found < 0 && hit) {
      found = 255 - (lane * 8 + e);
      fb = before;
    }
    before = after;
  }
  const unsigned ballot = __ballot_sync(FULL_MASK, found >= 0);
  if (ballot == 0) {
    if (lane == 0) { sm.sel_bin = -1; sm.sel_before = 0; }
    return;
  }
  const int src = __ffs(ballot) - 1;
  const int fbin = __shfl_sync(FULL_MASK, found, src);
  const unsigned long long fbefore = __shfl_sync(FULL_MASK, fb, src);
  if (lane == 0) { sm.sel_bin = fbin; sm.sel_before = fbefore; }
}

template <typename T>
__global__ void __launch_bounds__(kSampThreads, 1)
sample_kernel(int32_t* __restrict__ token_ids, const T* __restrict__ logits, int V, int64_t row_stride,
              bool vec_ok, const float* __restrict__ temperature, const int32_t* __restrict__ top_k,
              const float* __restrict__ top_p, const uint64_t* __restrict__ seeds,
              const uint64_t* __restrict__ offsets) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SampSmem& sm = *reinterpret_cast<SampSmem*>(smem_raw);
  using K = Keys<T>;
  constexpr int KB = K::BITS;
  const int r = blockIdx.x;
  const T* row = logits + (int64_t)r * row_stride;
  const int copy = (threadIdx.x >> 5) & (kHistCopies - 1);

  // ---- 1. max key, lowest index among maxima
  unsigned long long best = 0;
  for_each_elem<T>(row, V, vec_ok, [&](int j, uint32_t b) {
    const unsigned long long pk = ((unsigned long long)K::key(b) << 32) | (0xffffffffu - (uint32_t)j);
    best = pk > best ? pk : best;
  });
  best = block_max_u64(best, sm.red);
  const uint32_t kmax = (uint32_t)(best >> 32);
  const int imax = (int)(0xffffffffu - (uint32_t)(best & 0xffffffffu));
  const float T_ = temperature[r];
  if (!(T_ > 0.f)) {
    if (threadIdx.x == 0) token_ids[r] = imax;
    return;
  }
  const float m = K::value_of_key(kmax);
  const float log2e_over_T = 1.4426950408889634f / T_;

  // ---- 2. top-k threshold key (exactly k kept)
  const int k = top_k[r];
  const bool topk_on = k > 0 && k < V;
  uint32_t kth = 0;          // key of the k-th largest
  int need_eq = 0, cnt_eq = 0;
  if (topk_on) {
    uint32_t prefix = 0;
    unsigned long long remaining = (unsigned long long)k;
    for (int shift = KB - 8; shift >= 0; shift -= 8) {
      hist_clear(sm);
      __syncthreads();
      const uint32_t hi_mask = (shift + 8 >= 32) ? 0u : (~0u << (shift + 8));
      for_each_elem<T>(row, V, vec_ok, [&](int, uint32_t b) {
        const uint32_t key = K::key(b);
        if ((key & hi_mask) == (prefix & hi_mask))
          atomicAdd(reinterpret_cast<unsigned int*>(&sm.hist[copy][(key >> shift) & 255u]), 1u);
      });
      __syncthreads();
      if (threadIdx.x < 256) {
        unsigned long long s = 0;
#pragma unroll
        for (int c = 0; c < kHistCopies; ++c)
          s += (unsigned int)(sm.hist[c][threadIdx.x] & 0xffffffffull);
        sm.tot[threadIdx.x] = s;
      }
      __syncthreads();
      select_bin(sm, remaining, false);
      __syncthreads();
      const int bin = sm.sel_bin;
      remaining -= sm.sel_before;
      prefix |= (uint32_t)bin << shift;
      if (shift == 0) cnt_eq = (int)sm.tot[bin];
      __syncthreads();
    }
    kth = prefix;
    need_eq = (int)remaining;
  }

  // fixed-point weight of a value: exp((x - m) / T) * 2^40, rounded
  auto wfix = [&](float x) -> unsigned long long {
    const float w = exp2f((x - m) * log2e_over_T);
    return __float2ull_rn(w * 1099511627776.0f);
  };

  // ---- 3. nucleus threshold key tau (keep key >= tau)
  const float p = top_p[r];
  uint32_t tau = 0;
  if (p < 1.f) {
    uint32_t prefix = 0;
    unsigned long long target = 0, above = 0;
    bool done = false;
    for (int shift = KB - 8; shift >= 0 && !done; shift -= 8) {
      hist_clear(sm);
      __syncthreads();
      const uint32_t hi_mask = (shift + 8 >= 32) ? 0u : (~0u << (shift + 8));
      for_each_elem<T>(row, V, vec_ok, [&](int, uint32_t b) {
        const uint32_t key = K::key(b);
        if ((key & hi_mask) != (prefix & hi_mask)) return;
        if (topk_on && key <= kth) return;     // ties at the k-th key added below
        atomicAdd(&sm.hist[copy][(key >> shift) & 255u], wfix(K::value(b)));
      });
      __syncthreads();
      if (threadIdx.x == 0 && topk_on && need_eq > 0 && (kth & hi_mask) == (prefix & hi_mask))
        sm.hist[0][(kth >> shift) & 255u] += (unsigned long long)need_eq * wfix(K::value_of_key(kth));
      __syncthreads();
      hist_total(sm);
      __syncthreads();
      if (shift == KB - 8) {
        unsigned long long Z = 0;
        for (int b = 0; b < 256; ++b) Z += sm.tot[b];   // same value in every thread
        target = (unsigned long long)((double)p * (double)Z);
      }
      select_bin(sm, target - above, true);
      __syncthreads();
      const int bin = sm.sel_bin;
      if (bin < 0) {
        prefix = 0;          // the whole set is needed to exceed p: keep all
        done = true;
      } else {
        above += sm.sel_before;
        prefix |= (uint32_t)bin << shift;
      }
      __syncthreads();
    }
    tau = prefix;
  }

  // ---- 4. Gumbel-max over the kept ids
  const uint64_t seed = seeds[r], off = offsets[r];
  const float span = -kGumbelSpan;
  unsigned long long win = 0;
  auto consider = [&](int j, uint32_t b, bool tie_ok) {
    const uint32_t key = K::key(b);
    if (key < tau) return;
    if (topk_on && (key < kth || (key == kth && !tie_ok))) return;
    const float x = K::value(b);
    if ((x - m) * (1.f / T_) < span) return;
    const float score = __fdiv_rn(x, T_) + gumbel_noise(seed, off, (uint32_t)j);
    const unsigned long long pk = ((unsigned long long)f32_order_key(score) << 32) | (0xffffffffu - (uint32_t)j);
    win = pk > win ? pk : win;
  };
  // ties at the k-th key straddle the cut: keep the need_eq lowest indices,
  // i.e. those <= the need_eq-th smallest index of the tie group (radix
  // select on 24-bit inverted indices, counting tie elements only)
  const bool need_rank = topk_on && need_eq < cnt_eq;
  uint32_t tie_cut = 0xffffffffu;
  if (need_rank) {
    uint32_t prefix = 0;
    unsigned long long remaining = (unsigned long long)need_eq;
    for (int shift = 16; shift >= 0; shift -= 8) {
      hist_clear(sm);
      __syncthreads();
      const uint32_t hi_mask = (shift + 8 >= 24) ? 0u : ((~0u << (shift + 8)) & 0xffffffu);
      for_each_elem<T>(row, V, vec_ok, [&](int j, uint32_t b) {
        if (K::key(b) != kth) return;
        const uint32_t ik = 0xffffffu - (uint32_t)j;
        if ((ik & hi_mask) == (prefix & hi_mask))
          atomicAdd(reinterpret_cast<unsigned int*>(&sm.hist[copy][(ik >> shift) & 255u]), 1u);
      });
      __syncthreads();
      if (threadIdx.x < 256) {
        unsigned long long s = 0;
#pragma unroll
        for (int c = 0; c < kHistCopies; ++c)
          s += (unsigned int)(sm.hist[c][threadIdx.x] & 0xffffffffull);
        sm.tot[threadIdx.x] = s;
      }
      __syncthreads();
      select_bin(sm, remaining, false);
      __syncthreads();
      remaining -= sm.sel_before;
      prefix |= (uint32_t)sm.sel_bin << shift;
      __syncthreads();
    }
    tie_cut = 0xffffffu - prefix;
  }
  for_each_elem<T>(row, V, vec_ok, [&](int j, uint32_t b) { consider(j, b, (uint32_t)j <= tie_cut); });
  win = block_max_u64(win, sm.red);
  if (threadIdx.x == 0) {
    token_ids[r] = win ? (int)(0xffffffffu - (uint32_t)(win & 0xffffffffull)) : imax;
  }
}

cudaError_t launch_sample(int32_t* token_ids, const void* logits, int dtype, int num_rows, int vocab,
                          int64_t row_stride, const float* temperature, const int32_t* top_k,
                          const float* top_p, const uint64_t* seeds, const uint64_t* offsets,
                          cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  const int esz = dtype == PKVD_F32 ? 4 : 2;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && ((row_stride * esz) % 16 == 0);
  const size_t smem = sizeof(SampSmem);
  cudaError_t e = cudaSuccess;
#define PKVD_LAUNCH_SAMPLE(TYPE)                                                                     \
  do {                                                                                               \
    static bool configured = false;                                                                  \
    if (!configured) {                                                                               \
      e = cudaFuncSetAttribute(sample_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                               (int)smem);                                                           \
      if (e != cudaSuccess) return e;                                                                \
      configured = true;                                                                             \
    }                                                                                                \
    sample_kernel<TYPE><<<num_rows, kSampThreads, smem, stream>>>(                                   \
        token_ids, static_cast<const TYPE*>(logits), vocab, row_stride, vec_ok, temperature, top_k,  \
        top_p, seeds, offsets);                                                                      \
  } while (0)
  if (dtype == PKVD_F32) PKVD_LAUNCH_SAMPLE(float);
  else if (dtype == PKVD_F16) PKVD_LAUNCH_SAMPLE(__half);
  else PKVD_LAUNCH_SAMPLE(__nv_bfloat16);
#undef PKVD_LAUNCH_SAMPLE
  return cudaGetLastError();
}

}  // namespace pkvd
