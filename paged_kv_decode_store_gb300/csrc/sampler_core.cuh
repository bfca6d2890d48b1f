// Fused decode sampler: temperature, top-k, nucleus cut, Gumbel-max draw.
// (The kernel and its launcher; sampler.cu and sampler512.cu each build it
// once, with CTAs of PKVD_SAMP_THREADS threads, in namespace PKVD_SAMP_NS.)
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
// GB300 design -- no sort, one read of the row from HBM:
// * A row is split over a cluster of CS CTAs (CS = 1..8, chosen so the grid
//   covers the SMs).  Each CTA copies its slice into shared memory with
//   cp.async.bulk (TMA engine) and every later pass reads shared memory.
//   Row-wide values (max, histograms, the winning score) are exchanged
//   through distributed shared memory (mapa / ld.shared::cluster) between
//   cluster barriers, summed in rank order so results are deterministic.
// * Order-preserving integer keys of the raw logits (16-bit keys for
//   fp16/bf16) make top-k exact.  For 16-bit logits a key is one value, so
//   exact per-key counts in a window of keys below the max give each key's
//   probability mass as count * w(key), w in 2^-40 fixed point; ids below
//   the window only enter the normaliser, through an f32 sum in fixed order.
//   Top-k and the nucleus cut are found by walking that window down from
//   the max, two bins per thread and step; the window is counted in two stages (the
//   first 2048 keys, then the rest only when a cut lies deeper).  fp32
//   logits, and cuts that fall below the window, use an MSB-first radix
//   select with cluster-summed histograms instead.
// * Gumbel pass: only ids that can win are considered (x'_j >= max x' - 21,
//   since u lies in [2^-24, 1 - 2^-24] and g in [-2.81, 16.64]).  For 16-bit
//   logits the candidates are compacted into one list per CTA (in no
//   particular order: the race is a max of keys that carry the id) and
//   scored evenly by all threads; the generic path queues them per warp.
//   Either way Philox and the logarithms run on full warps.
// * Ties at the k-th key straddling the cut: slices are ordered by index, so
//   each CTA takes its share of the lowest-index ties.  For 16-bit logits the
//   shares come from the window bins and the one CTA whose share ends inside
//   its ties finds that tie by a block scan of per-thread runs; the generic
//   path resolves its share with a local radix select over its tie indices.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "device_cache.h"
#include "launch.h"

#ifndef PKVD_SAMP_THREADS
#error "define PKVD_SAMP_THREADS (1024 or 512) and PKVD_SAMP_NS before including this file"
#endif

namespace pkvd {
namespace PKVD_SAMP_NS {


constexpr int kSampThreads = PKVD_SAMP_THREADS;   // threads of one CTA (this build of the kernel)
constexpr int kSampCtasPerSm = 1024 / kSampThreads;   // CTAs an SM holds at once (64 registers a thread)
// shared memory of one CTA: the SM's 228 KB shared by kSampCtasPerSm CTAs,
// less the 1 KB the hardware reserves per CTA
constexpr int kSampSmem = (233472 / kSampCtasPerSm) - 1024;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kHistCopies = 16;
constexpr float kGumbelSpan = 21.0f;
constexpr int kMaxCluster = 8;
constexpr int kMaxChunks = 16;
constexpr int kChunkBytes = 16 * kSampThreads;   // one 16-byte word per thread
static_assert(kChunkBytes / 16 == kSampThreads, "one 16-byte word per thread and chunk");
constexpr int kQueue = 64;                 // per-warp candidate ring

// Exact per-key counts are kept for the kWinTop keys below the row max
// (16-bit logits: 8 binades for fp16, 64 for bf16).
constexpr int kWinTop = 8192;                   // exact counts of the top keys below the max
constexpr int kWinBlock = 2 * kSampThreads;     // bins per walk step (two per thread)
// First counting stage: the keys of the two binades below the max (fp16 has
// 1024 keys per binade, bf16 128).
template <typename T>
constexpr int win1_bins() { return std::is_same<T, __half>::value ? 2048 : 256; }

template <typename T> struct Keys;
template <> struct Keys<float> {
  static constexpr int BITS = 32;
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

__device__ __forceinline__ uint32_t f32_order_key(float x) { return Keys<float>::key(__float_as_uint(x)); }

// ------------------------------------------------------------- cluster PTX
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split cluster barrier: every thread arrives once at kernel start and waits
// before its CTA's first access to a peer's shared memory, which is how a
// CTA knows that every CTA of its cluster has started.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ unsigned int dsmem_ld_u32(uint32_t a) {
  unsigned int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long dsmem_ld_u64(uint32_t a) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}

// ---------------------------------------------------------------- Philox
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

// 2^x on the special-function unit with results below 2^-126 flushed to
// zero (each such term is under 2^-126 of the max term, which is 1)
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// E_j = -ln u_j for id j's uniform: word (j mod 4) of Philox4x32-10 at
// counter (j / 4, offset), u = ((w >> 9) + 1/2) 2^-23, exact in f32 and
// strictly inside (0, 1), so E_j > 0 (accurate near u = 1, where it is tiny)
__device__ __forceinline__ float noise_of_word(uint32_t w) {
  const float u = (__uint2float_rn(w >> 9) + 0.5f) * 1.1920928955078125e-07f;   // * 2^-23, exact
  return -logf(u);
}
// The four Philox words of ids 4c .. 4c + 3 (one call serves the four).
__device__ __forceinline__ uint4 noise_words(uint64_t seed, uint64_t offset, uint32_t c) {
  const uint4 ctr = make_uint4(c, (uint32_t)offset, (uint32_t)(offset >> 32), 0u);
  return philox4x32_10(ctr, make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}
__device__ __forceinline__ float exp_noise(uint64_t seed, uint64_t offset, uint32_t j) {
  const uint4 w4 = noise_words(seed, offset, j >> 2);
  const uint32_t sel = j & 3u;
  return noise_of_word(sel == 0 ? w4.x : (sel == 1 ? w4.y : (sel == 2 ? w4.z : w4.w)));
}

// Gumbel-max as an exponential race: argmax_j x_j / T - ln(-ln u_j) is
// argmin_j E_j exp((m - x_j) / T) for any m; with m the row max (or a bound
// above every x_j of the slice) the factor lies in [1, 2^31) for every id
// that can win.  The packed key makes the smallest race time the largest
// key, and the lowest id the winner among equal times.  d2 = (m - x) / (T ln 2).
__device__ __forceinline__ unsigned long long race_key_of(float e, uint32_t j, float d2) {
  const float t = e * ex2_ftz(d2);
  return ((unsigned long long)(uint32_t)~f32_order_key(t) << 32) | (0xffffffffu - j);
}
__device__ __forceinline__ unsigned long long race_key(uint64_t seed, uint64_t offset, uint32_t j, float d2) {
  return race_key_of(exp_noise(seed, offset, j), j, d2);
}

// ------------------------------------------------------------ shared state
struct SampHdr {
  ulonglong2 px[2][kMaxCluster];          // pushed cluster exchanges (alternating)
  uint64_t bar[kMaxChunks];
  int gap[kMaxCluster];                  // row max key - each rank's max key
  unsigned long long ex_arr[2][256];     // cluster-exchanged arrays (alternating)
  unsigned long long tot[256];           // row-wide totals of the last exchange
  unsigned long long red[kSampWarps];
  int sel_bin;
  unsigned long long sel_before;
  int sel_aux;
  unsigned long long sel_val;
  unsigned long long zsum;
  unsigned int tie_mine;                 // this CTA's count of the k-th key
  long long tie_before;                  // that count over the lower ranks
  unsigned long long fin_best;           // the row's winning race key (warp 0's combine of the ranks)
  float fin_mm;                          // the largest rank bound
  uint32_t fin_tie;                      // the last kept tie over the ranks
};

struct Ctx {
  SampHdr* h;
  int cs;        // cluster size
  int ex;        // next exchange slot
};

// Cluster exchange of two u64 per CTA: threads 0..cs-1 store this CTA's
// pair into slot [rank] of every CTA's table (its own included), then one
// cluster barrier; afterwards every rank's pair is in local shared memory
// and no CTA reads a peer after the barrier.  Consecutive exchanges use
// alternate tables: a peer can only write a table again after the next
// barrier, which every reader of the previous values has reached.
// v0 and v1 must be uniform over the block.
__device__ __forceinline__ const ulonglong2* cluster_push(Ctx& c, uint32_t crank, unsigned long long v0,
                                                          unsigned long long v1) {
  const int s = c.ex;
  c.ex ^= 1;
  if (threadIdx.x < (unsigned)c.cs) {
    const uint32_t addr = dsmem_addr(&c.h->px[s][crank], threadIdx.x);
    asm volatile("st.shared::cluster.v2.u64 [%0], {%1, %2};" ::"r"(addr), "l"(v0), "l"(v1) : "memory");
  }
  cluster_sync();
  return c.h->px[s];
}

// Max or sum of a block-uniform u64 over the cluster, in rank order.
template <bool MAX>
__device__ __forceinline__ unsigned long long cluster_scalar(Ctx& c, unsigned long long v) {
  const ulonglong2* px = cluster_push(c, cluster_rank(), v, 0ull);
  unsigned long long acc = 0;
  for (int r = 0; r < c.cs; ++r) {
    const unsigned long long x = px[r].x;
    acc = MAX ? (x > acc ? x : acc) : acc + x;
  }
  return acc;
}

// Sum the 256-entry arrays every CTA wrote to ex_arr[c.ex] into tot[].
// Threads 0..255 own one entry each; ends with __syncthreads.
__device__ __forceinline__ void cluster_sum_array(Ctx& c) {
  const int s = c.ex;
  c.ex ^= 1;
  cluster_sync();
  if (threadIdx.x < 256) {
    unsigned long long acc = 0;
    for (int r = 0; r < c.cs; ++r) acc += dsmem_ld_u64(dsmem_addr(&c.h->ex_arr[s][threadIdx.x], r));
    c.h->tot[threadIdx.x] = acc;
  }
  __syncthreads();
}

// Block-wide max / sum / exclusive scan of a u64 per thread.  Warp partials
// go through s[0..kSampWarps); every warp then reduces them with shuffles
// (lanes past the last warp contribute zero), so two barriers suffice.  The first barrier also protects s[]
// from the previous user; none of these ends with a barrier.
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
  v = lane < kSampWarps ? s[lane] : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(FULL_MASK, v, o);
    v = t > v ? t : v;
  }
  return v;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  v = lane < kSampWarps ? s[lane] : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v, unsigned long long* s,
                                                                  unsigned long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) s[warp] = incl;
  __syncthreads();
  const unsigned long long x = lane < kSampWarps ? s[lane] : 0ull;
  unsigned long long xin = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(FULL_MASK, xin, o);
    if (lane >= o) xin += t;
  }
  total = __shfl_sync(FULL_MASK, xin, 31);
  const unsigned long long wbase = __shfl_sync(FULL_MASK, xin - x, warp);
  return wbase + incl - v;
}

// Warp 0 walks tot[] (descending bin order if DESC) and finds the first bin
// where before + tot[b] crosses target (>= for counts, > for mass).
// sel_bin = -1 if none; ends with __syncthreads.
template <bool DESC>
__device__ __forceinline__ void select_bin(SampHdr& h, unsigned long long target, bool strict) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned long long v[8], local = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int b = lane * 8 + e;
      v[e] = h.tot[DESC ? 255 - b : b];
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
      if (found < 0 && (strict ? after > target : after >= target)) {
        const int b = lane * 8 + e;
        found = DESC ? 255 - b : b;
        fb = before;
      }
      before = after;
    }
    const unsigned ballot = __ballot_sync(FULL_MASK, found >= 0);
    if (ballot == 0) {
      if (lane == 0) { h.sel_bin = -1; h.sel_before = 0; }
    } else {
      const int src = __ffs(ballot) - 1;
      const int fbin = __shfl_sync(FULL_MASK, found, src);
      const unsigned long long fbefore = __shfl_sync(FULL_MASK, fb, src);
      if (lane == 0) { h.sel_bin = fbin; h.sel_before = fbefore; }
    }
  }
  __syncthreads();
}

// round(w * 2^40) for w in [0, 1], built from the float's bits (no 64-bit
// float conversion, which runs on the slow fp64 pipe of this part).
__device__ __forceinline__ unsigned long long fixed_weight(float w) {
  const uint32_t b = __float_as_uint(w);
  const int ex = (int)((b >> 23) & 0xffu);
  if (ex == 0) return 0ull;
  const unsigned long long man = (b & 0x7fffffu) | 0x800000u;
  const int sh = ex - 127 + 40 - 23;
  if (sh >= 0) return man << sh;
  if (sh < -24) return 0ull;
  return (man + (1ull << (-sh - 1))) >> (-sh);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}

// Warp 0: first entry i of tot[0..N) (ascending) where base + tot[0..i]
// crosses target (>= if !strict, > if strict).  Writes sel_bin = i (-1 if
// none), sel_before = base + tot[0..i), sel_aux = tot[i]; ends with __syncthreads.
template <int N>
__device__ __forceinline__ void find_first(SampHdr& h, unsigned long long base, unsigned long long target,
                                           bool strict) {
  constexpr int PER = N / 32;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned long long v[PER], local = 0;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      v[e] = h.tot[lane * PER + e];
      local += v[e];
    }
    unsigned long long incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += t;
    }
    unsigned long long before = base + incl - local;
    int found = -1;
    unsigned long long fb = 0, fv = 0;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const unsigned long long after = before + v[e];
      if (found < 0 && (strict ? after > target : after >= target)) {
        found = lane * PER + e;
        fb = before;
        fv = v[e];
      }
      before = after;
    }
    const unsigned ballot = __ballot_sync(FULL_MASK, found >= 0);
    if (ballot == 0) {
      if (lane == 0) { h.sel_bin = -1; h.sel_before = 0; h.sel_val = 0; }
    } else {
      const int src = __ffs(ballot) - 1;
      const int fi = __shfl_sync(FULL_MASK, found, src);
      const unsigned long long b2 = __shfl_sync(FULL_MASK, fb, src);
      const unsigned long long v2 = __shfl_sync(FULL_MASK, fv, src);
      if (lane == 0) { h.sel_bin = fi; h.sel_before = b2; h.sel_val = v2; }
    }
  }
  __syncthreads();
}

// Warp 0 sums tot[0..256) into h.zsum; ends with __syncthreads.
__device__ __forceinline__ unsigned long long sum_tot(SampHdr& h) {
  if (threadIdx.x < 32) {
    unsigned long long s = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) s += h.tot[threadIdx.x * 8 + e];
    s = warp_sum_u64(s);
    if (threadIdx.x == 0) h.zsum = s;
  }
  __syncthreads();
  return h.zsum;
}

// Visit the CTA's elements: f(local index, raw bits).  `src` is shared or
// global memory; 16-byte vectors when aligned.
template <typename T, typename F>
__device__ __forceinline__ void visit(const T* src, int n, bool vec, F&& f) {
  constexpr int E = 16 / sizeof(T);
  int done = 0;
  if (vec) {
    const int nv = n / E;
    const uint4* sv = reinterpret_cast<const uint4*>(src);
    for (int v = threadIdx.x; v < nv; v += kSampThreads) {
      const uint4 u = sv[v];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint32_t b = (sizeof(T) == 4) ? w[e] : ((w[e / 2] >> (16 * (e & 1))) & 0xffffu);
        f(v * E + e, b);
      }
    }
    done = nv * E;
  }
  for (int j = done + threadIdx.x; j < n; j += kSampThreads)
    f(j, sizeof(T) == 4 ? __float_as_uint(*reinterpret_cast<const float*>(src + j))
                        : (uint32_t)(*reinterpret_cast<const unsigned short*>(src + j)));
}

struct SampArgs {
  int fast;             // 16-bit keys, resident slice: windowed path
  int list_cap;         // fast path: list entries after the first window's bins
  int32_t* token_ids;
  const void* logits;
  int V;
  int64_t row_stride;
  int slice;            // elements per CTA (a multiple of 16 bytes)
  int resident;         // slice held in shared memory
  int vec;              // 16-byte aligned rows
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const uint64_t* seeds;
  const uint64_t* offsets;
  const uint32_t* mask;   // optional allowed-id bits [rows, mask_stride words] (bit j % 32 of word j / 32)
  int64_t mask_stride;
  int32_t* row_info;      // optional per-row cut parameters for the extras kernel (kRowInfo ints)
};

template <typename T>
constexpr int region_bytes() {
  constexpr int w = sizeof(T) == 2 ? kWinTop * 4 : 0;
  constexpr int hst = kHistCopies * 256 * 8;
  constexpr int q = kSampWarps * kQueue * 8;
  return (w > hst ? (w > q ? w : q) : (hst > q ? hst : q));
}

// Order-preserving keys of the two 16-bit floats of a word, in one go:
// -0 is first folded onto +0, then key = b ^ 0xffff (negative) or b ^ 0x8000.
// Two 16-bit floats of one 32-bit word, as the packed type of T.
template <typename T> struct Pack2;
template <> struct Pack2<__half> {
  using T2 = __half2;
  static constexpr uint32_t kNegInf2 = 0xfc00fc00u;
  __device__ static float2 to_float2(uint32_t w) { return __half22float2(*reinterpret_cast<const __half2*>(&w)); }
};
template <> struct Pack2<__nv_bfloat16> {
  using T2 = __nv_bfloat162;
  static constexpr uint32_t kNegInf2 = 0xff80ff80u;
  __device__ static float2 to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
};
template <typename T>
__device__ __forceinline__ typename Pack2<T>::T2 as_t2(uint32_t w) {
  return *reinterpret_cast<const typename Pack2<T>::T2*>(&w);
}
template <typename T>
__device__ __forceinline__ uint32_t t2_bits(typename Pack2<T>::T2 v) {
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t keys2(uint32_t w) {
  const uint32_t nz = ((w & 0x7fff7fffu) + 0x7fff7fffu) & 0x80008000u;   // magnitude != 0, per half
  w &= nz | 0x7fff7fffu;
  const uint32_t s = (w >> 15) & 0x00010001u;
  return w ^ ((s * 0x7fffu) | 0x80008000u);
}

// Masked ids become -inf: weight 0 in every sum, below every allowed id in
// every cut, never a candidate while an allowed id remains.  `bits` holds
// the 8 allowed bits of the word's 8 logits (bit e for logit e).
template <typename T>
__device__ __forceinline__ uint4 apply_mask16(uint4 u, uint32_t bits) {
  constexpr uint32_t ninf = Pack2<T>::kNegInf2;
  auto one = [&](uint32_t w, uint32_t b2) {
    const uint32_t keep = ((b2 & 1u) ? 0x0000ffffu : 0u) | ((b2 & 2u) ? 0xffff0000u : 0u);
    return (w & keep) | (ninf & ~keep);
  };
  u.x = one(u.x, bits);
  u.y = one(u.y, bits >> 2);
  u.z = one(u.z, bits >> 4);
  u.w = one(u.w, bits >> 6);
  return u;
}
__device__ __forceinline__ bool allowed_bit(const uint32_t* bits, int64_t j) {
  return (bits[j >> 5] >> (j & 31)) & 1u;
}
template <typename T> __device__ __forceinline__ T neg_inf_value();
template <> __device__ __forceinline__ float neg_inf_value<float>() { return __uint_as_float(0xff800000u); }
template <> __device__ __forceinline__ __half neg_inf_value<__half>() { return __ushort_as_half((unsigned short)0xfc00u); }
template <> __device__ __forceinline__ __nv_bfloat16 neg_inf_value<__nv_bfloat16>() {
  return __ushort_as_bfloat16((unsigned short)0xff80u);
}

// Eight bits, one per logit of a 16-byte word of 16-bit floats (bit e for
// logit e), set where the value is >= the threshold value held in both
// halves of t.  A value compare is the same test as a key compare.
template <typename T>
__device__ __forceinline__ uint32_t pass_bits(const uint4 u, const typename Pack2<T>::T2 t) {
  const uint32_t g0 = __hge2_mask(as_t2<T>(u.x), t), g1 = __hge2_mask(as_t2<T>(u.y), t);
  const uint32_t g2 = __hge2_mask(as_t2<T>(u.z), t), g3 = __hge2_mask(as_t2<T>(u.w), t);
  const uint32_t lo4 = (g0 & 0x00010001u) | ((g1 & 0x00010001u) << 2) | ((g2 & 0x00010001u) << 4) |
                       ((g3 & 0x00010001u) << 6);
  // bits 0,2,4,6 hold the low halves, bits 16,18,20,22 the high halves
  return (lo4 & 0x55u) | ((lo4 >> 15) & 0xaau);
}

// Threshold value of a 16-bit key, in both halves of a word (-inf for key 0,
// which every value reaches).
template <typename T>
__device__ __forceinline__ typename Pack2<T>::T2 key_threshold2(uint32_t key) {
  const uint32_t tb = key == 0 ? (Pack2<T>::kNegInf2 & 0xffffu) : ((key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu));
  return as_t2<T>(tb | (tb << 16));
}

// Add one to win[d] for every id of a resident 16-bit slice whose key lies
// at distance d in [d_lo, d_lo + width) below kmax (every key <= kmax).
template <typename T>
__device__ __forceinline__ void count_bins16(const uint4* sv, int nvec, int rest, int n, const T* slice,
                                             uint32_t kmax, uint32_t* win, uint32_t d_lo, uint32_t width) {
  const uint32_t kmax2 = kmax | (kmax << 16);
  for (int v = threadIdx.x; v < nvec; v += kSampThreads) {
    const uint4 u = sv[v];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // per-half kmax - key: no borrow crosses the halves, as every key <= kmax
      const uint32_t d2 = kmax2 - keys2(w[q]);
      const uint32_t dl = (d2 & 0xffffu) - d_lo, dh = (d2 >> 16) - d_lo;
      if (dl < width) atomicAdd(&win[d_lo + dl], 1u);
      if (dh < width) atomicAdd(&win[d_lo + dh], 1u);
    }
  }
  for (int j = rest + threadIdx.x; j < n; j += kSampThreads) {
    const uint32_t d = kmax - Keys<T>::key((uint32_t)(*reinterpret_cast<const unsigned short*>(slice + j))) - d_lo;
    if (d < width) atomicAdd(&win[d_lo + d], 1u);
  }
}



template <typename T>
__global__ void __launch_bounds__(kSampThreads, kSampCtasPerSm) sample_kernel(const SampArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  using K = Keys<T>;
  constexpr int KB = K::BITS;
  constexpr int E = 16 / sizeof(T);
  SampHdr& h = *reinterpret_cast<SampHdr*>(smem_raw);
  // [header][resident slice][region]; the region is reused: window counts
  // and candidate lists, radix bins, Gumbel queues
  T* slice_smem = reinterpret_cast<T*>(smem_raw + ((sizeof(SampHdr) + 127) / 128) * 128);
  uint8_t* region = reinterpret_cast<uint8_t*>(slice_smem) +
                    (a.resident ? (((size_t)a.slice * sizeof(T) + 127) / 128) * 128 : 0);
  unsigned long long (*hist)[256] = reinterpret_cast<unsigned long long (*)[256]>(region);
  uint32_t* q_idx = reinterpret_cast<uint32_t*>(region);
  float* q_x = reinterpret_cast<float*>(region + kSampWarps * kQueue * 4);

  pdl_wait();                       // logits and parameters may come from the previous kernel
  pdl_trigger();
  cluster_arrive_relaxed();         // matched by cluster_wait() before the first peer access
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Ctx c{&h, (int)cluster_size(), 0};
  const uint32_t crank = cluster_rank();
  const int row_id = blockIdx.x / c.cs;
  const T* row = static_cast<const T*>(a.logits) + (int64_t)row_id * a.row_stride;
  const int lo = (int)crank * a.slice;
  const int n = max(0, min(a.V, lo + a.slice) - lo);
  const int copy = warp & (kHistCopies - 1);
  const uint32_t* mask_row = a.mask ? a.mask + (int64_t)row_id * a.mask_stride : nullptr;
  const uint64_t seed = a.seeds[row_id], off = a.offsets[row_id];
  // the row's sampling parameters, read before the slice lands so their
  // latency hides under the logit copies
  const float row_T = a.temperature[row_id], row_p = a.top_p[row_id];
  const int row_k = a.top_k[row_id];
  // the row's cut parameters for the extras kernel (rank 0 writes them)
  auto put_row_info = [&](int flags, uint32_t tau_k, uint32_t kth_k, uint32_t tie_enc, float row_max) {
    if (a.row_info && crank == 0 && tid == 0) {
      int32_t* ri = a.row_info + (int64_t)row_id * kRowInfo;
      ri[0] = flags;
      ri[1] = (int32_t)tau_k;
      ri[2] = (int32_t)kth_k;
      ri[3] = tie_enc == 0xffffffffu ? 0x7fffffff : (int32_t)tie_enc - 1;   // last kept tie at the k-th key
      ri[4] = __float_as_int(row_max);
    }
  };
  // a tie candidate in 32 bits for a max over ranks (INT_MAX -> all ones)
  auto tie_code = [](int cand) -> uint32_t { return cand == 0x7fffffff ? 0xffffffffu : (uint32_t)(cand + 1); };
  // No candidate anywhere (every id masked, or no finite logit): every id
  // counts the same, so the race is over -ln u alone.  Returns the row's best
  // packed (race key, ~id); cluster-uniform.
  auto uniform_draw = [&]() -> unsigned long long {
    unsigned long long ub = 0;
    for (int j = tid; j < n; j += kSampThreads) {
      const unsigned long long pk = race_key(seed, off, (uint32_t)(lo + j), 0.f);
      ub = pk > ub ? pk : ub;
    }
    ub = block_max_u64(ub, h.red);
    return cluster_scalar<true>(c, ub);
  };

  if constexpr (sizeof(T) == 2) {
    if (a.fast) {
      // ================= 16-bit logits, resident slice
      constexpr int kWin1 = win1_bins<T>();
      using T2 = typename Pack2<T>::T2;
      const uint4* sv = reinterpret_cast<const uint4*>(slice_smem);
      const int nvec = n / 8;
      const int rest = nvec * 8;
      auto bits_at = [&](int j) -> uint32_t {
        return (uint32_t)(*reinterpret_cast<const unsigned short*>(slice_smem + j));
      };
      // ---- F0 + F1. slice -> shared memory in 16 KB bulk copies; each
      // thread folds its word of a chunk into a packed max (one instruction
      // per two logits) as soon as the chunk lands
      T2 mx2 = as_t2<T>(Pack2<T>::kNegInf2);
      {
        const int bulk = nvec * 16;
        const int nch = (bulk + kChunkBytes - 1) / kChunkBytes;
        // thread 0 sets up the barriers and issues every copy before the
        // CTA-wide barrier, so the requests leave while the other warps of
        // the CTA are still arriving; the barrier then publishes the
        // initialised mbarriers to the waiting threads
        if (tid == 0) {
          for (int i = 0; i < nch; ++i) mbar_init(&h.bar[i], 1);
          fence_mbar_init();
          for (int i = 0; i < nch; ++i) {
            const int off = i * kChunkBytes;
            const int sz = min(kChunkBytes, bulk - off);
            mbar_arrive_expect_tx(&h.bar[i], (uint32_t)sz);
            bulk_g2s(reinterpret_cast<uint8_t*>(slice_smem) + off, reinterpret_cast<const uint8_t*>(row + lo) + off,
                     (uint32_t)sz, &h.bar[i]);
          }
        }
        __syncthreads();
        for (int j = rest + tid; j < n; j += kSampThreads)
          slice_smem[j] = (mask_row && !allowed_bit(mask_row, lo + j)) ? neg_inf_value<T>() : row[lo + j];
        const uint8_t* mbytes = mask_row ? reinterpret_cast<const uint8_t*>(mask_row) + (lo >> 3) : nullptr;
        for (int i = 0; i < nch; ++i) {
          mbar_wait_bounded(&h.bar[i], 0);
          const int v = i * (kChunkBytes / 16) + tid;           // one 16-byte word per thread and chunk
          if (v < nvec) {
            uint4 u = sv[v];
            if (mbytes) {                                       // masked ids become -inf in place
              u = apply_mask16<T>(u, mbytes[v]);
              reinterpret_cast<uint4*>(slice_smem)[v] = u;
            }
            mx2 = __hmax2(mx2, __hmax2(__hmax2(as_t2<T>(u.x), as_t2<T>(u.y)), __hmax2(as_t2<T>(u.z), as_t2<T>(u.w))));
          }
        }
        __syncthreads();
      }
      uint32_t kmr;        // this CTA's max key
      {
        const uint32_t mw = t2_bits<T>(mx2);
        uint32_t mx = max(K::key(mw & 0xffffu), K::key(mw >> 16));
        for (int j = rest + tid; j < n; j += kSampThreads) mx = max(mx, K::key(bits_at(j)));
        kmr = (uint32_t)block_max_u64(mx, h.red);
      }
      cluster_wait();                                   // every peer has started
      const float Tr = row_T;
      if (!(Tr > 0.f)) {
        // greedy: this slice's lowest index holding its max key, then one
        // exchange; the packed (key, ~index) max is the row's answer
        uint32_t first = 0xffffffffu;
        const uint32_t km2 = kmr | (kmr << 16);
        for (int v = tid; v < nvec; v += kSampThreads) {
          const uint4 u = sv[v];
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t x2 = keys2(w[q]) ^ km2;
            if ((x2 & 0xffffu) == 0) first = min(first, (uint32_t)(v * 8 + q * 2));
            if ((x2 >> 16) == 0) first = min(first, (uint32_t)(v * 8 + q * 2 + 1));
          }
        }
        for (int j = rest + tid; j < n; j += kSampThreads)
          if (K::key(bits_at(j)) == kmr) first = min(first, (uint32_t)j);
        // the min index among the threads that saw the max key is the max of
        // its complement
        const unsigned long long mine =
            first == 0xffffffffu ? 0ull : (((unsigned long long)kmr << 32) | (0xffffffffull - (unsigned long long)(lo + (int)first)));
        const unsigned long long pk = block_max_u64(mine, h.red);
        const ulonglong2* px = cluster_push(c, crank, pk, 0ull);
        if (crank == 0 && tid == 0) {
          unsigned long long best = 0;
          for (int r = 0; r < c.cs; ++r) best = px[r].x > best ? px[r].x : best;
          a.token_ids[row_id] = (int)(0xffffffffu - (uint32_t)(best & 0xffffffffull));
        }
        put_row_info(kRowGreedy, 0u, 0u, 0u, 0.f);
        return;
      }
      const float l2t = 1.4426950408889634f / Tr;
      const int k = row_k;
      const bool topk_on = k > 0 && k < a.V;
      const float p = row_p;
      const bool nucleus_on = p < 1.f;
      const bool need_win = topk_on || nucleus_on;
      const bool need_z = nucleus_on && !topk_on;
      uint32_t kth = 0, tau = 0;
      long long need_eq = 0, cnt_eq = 0;
      bool topk_done = !topk_on, nucleus_done = !nucleus_on;
      uint32_t kmax = kmr;       // the row's max key (known after the window exchange)
      float m = K::value_of_key(kmr);
      bool list_ok = false;      // the list below holds every id of the first window
      bool windows_free = false; // no peer reads this CTA's window any more (cluster-uniform)
      int list_n = 0;

      // ---- F2. exact counts per key in a window of keys below the max.
      // Bins are distances from this CTA's own max key, so no exchange is
      // needed before counting; the walk shifts each peer's bins by the gap
      // between the row max and that peer's max.  Counting is staged: ids of
      // the first kWin1 keys are compacted into a list (count, block scan,
      // write) and binned from there in full warps, the normaliser Z of the
      // nucleus rides along the count pass (a compensated f32 sum per
      // thread, relative to this CTA's max, fixed point from there on); keys
      // down to kWinTop are counted straight from the slice only when a cut
      // lies that deep.
      uint32_t* win = reinterpret_cast<uint32_t*>(region);
      uint32_t* list = win + kWin1;
      if (need_win) {
        for (int i = tid; i < kWin1; i += kSampThreads) win[i] = 0u;
        const float mr = m;
        const float ml2t = mr * l2t;
        // packed test "key >= kmr - (kWin1 - 1)" on the values
        const uint32_t k1 = kmr >= (uint32_t)(kWin1 - 1) ? kmr - (uint32_t)(kWin1 - 1) : 0u;
        const T2 t1v2 = key_threshold2<T>(k1);
        float zs = 0.f, zc = 0.f;                 // compensated running sum
        auto zadd = [&](float y) {
          y -= zc;
          const float t = zs + y;
          zc = (t - zs) - y;
          zs = t;
        };
        // each word's pass mask is kept (one byte per word, at the far end
        // of the list's space) so that the write pass reads it instead of
        // comparing the word again; the list may use the space before it
        const int list_room = a.list_cap - (nvec + 3) / 4;
        uint8_t* wmask = reinterpret_cast<uint8_t*>(list + list_room);
        int hits = 0;
        for (int v = tid; v < nvec; v += kSampThreads) {
          const uint4 u = sv[v];
          const uint32_t cb = pass_bits<T>(u, t1v2);
          wmask[v] = (uint8_t)cb;
          hits += __popc(cb);
          if (need_z) {
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            float vs = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 f = Pack2<T>::to_float2(w[q]);
              vs += ex2_ftz(fmaf(f.x, l2t, -ml2t)) + ex2_ftz(fmaf(f.y, l2t, -ml2t));
            }
            zadd(vs);
          }
        }
        for (int j = rest + tid; j < n; j += kSampThreads) {
          const uint32_t b = bits_at(j);
          hits += K::key(b) >= k1;
          if (need_z) zadd(ex2_ftz((K::value(b) - mr) * l2t));
        }
        unsigned long long tot_u;
        const int first = (int)block_excl_scan_u64((unsigned long long)hits, h.red, tot_u);
        list_n = (int)tot_u;
        list_ok = list_n <= list_room;
        if (list_ok) {
          if (hits > 0) {
            int kk = first;
            for (int v = tid; v < nvec; v += kSampThreads) {
              uint32_t cb = wmask[v];
              while (cb) {
                const int e = __ffs(cb) - 1;
                cb &= cb - 1;
                list[kk++] = (uint32_t)(v * 8 + e);
              }
            }
            for (int j = rest + tid; j < n; j += kSampThreads)
              if (K::key(bits_at(j)) >= k1) list[kk++] = (uint32_t)j;
          }
          __syncthreads();
          for (int i = tid; i < list_n; i += kSampThreads) atomicAdd(&win[kmr - K::key(bits_at((int)list[i]))], 1u);
        } else {
          count_bins16<T>(sv, nvec, rest, n, slice_smem, kmr, win, 0u, (uint32_t)kWin1);
        }
        // one exchange: (max key, list flag) and Z relative to this CTA's
        // max; from here on every CTA's first window is final, so peers read
        // it in place over DSMEM
        const unsigned long long zr = block_sum_u64(need_z ? fixed_weight(zs) : 0ull, h.red);
        const ulonglong2* px = cluster_push(c, crank, ((unsigned long long)(list_ok ? 0u : 1u) << 32) | kmr, zr);
        for (int r = 0; r < c.cs; ++r) {
          kmax = max(kmax, (uint32_t)(px[r].x & 0xffffffffu));
          if (px[r].x >> 32) list_ok = false;
        }
        m = K::value_of_key(kmax);
        if (tid < c.cs) h.gap[tid] = (int)(kmax - (uint32_t)(px[tid].x & 0xffffffffu));
        if (tid == 0) {
          // Z = sum over ranks of Z_r * 2^((m_r - m) / T ln 2), each Z_r
          // relative to its rank's max (fp64 for the few products only)
          double zd = 0.0;
          if (need_z)
            for (int r = 0; r < c.cs; ++r)
              zd += (double)px[r].y * (double)exp2f((K::value_of_key((uint32_t)(px[r].x & 0xffffffffu)) - m) * l2t);
          h.zsum = (unsigned long long)zd;
        }
        __syncthreads();                                  // gap[] and zsum visible
        const unsigned long long zrow = h.zsum;
        auto wfix = [&](float x) -> unsigned long long { return fixed_weight(ex2_ftz((x - m) * l2t)); };
        int covered = kWin1;
        // the second stage: the bins it writes were never read (they held
        // the list), so peers may still be walking the first window
        // meanwhile; cluster-uniform
        auto widen = [&]() {
          __syncthreads();
          for (int i = kWin1 + tid; i < kWinTop; i += kSampThreads) win[i] = 0u;
          __syncthreads();
          count_bins16<T>(sv, nvec, rest, n, slice_smem, kmr, win, (uint32_t)kWin1, (uint32_t)(kWinTop - kWin1));
          cluster_sync();
          covered = kWinTop;
          list_ok = false;
        };

        // Walk the window down from the row max, kWinBlock bins per step
        // (two per thread); counts are the cluster sums of the bins, so
        // every CTA of the cluster takes the same branches.
        static_assert(kWinBlock == 2 * kSampThreads, "two bins per thread and walk step");
        // bins [d0, d1) of the row, d1 <= covered: every rank has counted
        // them (a rank's bin for row distance d is d - gap, below covered)
        auto row_counts = [&](int d0, int d1, unsigned int* cnt) {
          const int d = d0 + tid * 2;
          cnt[0] = cnt[1] = 0;
          for (int r = 0; r < c.cs; ++r) {
            const int dr = d - h.gap[r];               // the same key in rank r's bins
#pragma unroll
            for (int e = 0; e < 2; ++e)
              if (d + e < d1 && dr + e >= 0) cnt[e] += dsmem_ld_u32(dsmem_addr(&win[dr + e], (uint32_t)r));
          }
        };
        if (topk_on) {
          unsigned long long before = 0;
          for (int d0 = 0, d1 = 0; d0 < kWinTop && !topk_done; d0 = d1) {
            if (d0 >= covered) widen();
            d1 = min(d0 + kWinBlock, covered);
            unsigned int cnt[2];
            row_counts(d0, d1, cnt);
            const unsigned long long mine = (unsigned long long)cnt[0] + cnt[1];
            unsigned long long tot;
            unsigned long long acc = before + block_excl_scan_u64(mine, h.red, tot);
            if (acc < (unsigned long long)k && (unsigned long long)k <= acc + mine) {
              const int e = acc + cnt[0] >= (unsigned long long)k ? 0 : 1;
              h.sel_aux = d0 + tid * 2 + e;
              h.sel_before = e ? acc + cnt[0] : acc;
              h.sel_val = e ? cnt[1] : cnt[0];
            }
            __syncthreads();
            if (before + tot >= (unsigned long long)k) {
              kth = kmax - (uint32_t)h.sel_aux;
              need_eq = k - (long long)h.sel_before;
              cnt_eq = (long long)h.sel_val;
              topk_done = true;
            }
            before += tot;
          }
        }
        if (nucleus_on && topk_done) {
          const int dk = topk_on ? (int)(kmax - kth) : kWinTop;   // bins past the k-th key are out
          const unsigned long long tie_mass = topk_on ? (unsigned long long)need_eq * wfix(K::value_of_key(kth)) : 0ull;
          auto bin_mass = [&](int d, int d1, unsigned int cnt) -> unsigned long long {
            if (d >= d1 || d > dk) return 0ull;
            if (topk_on && d == dk) return tie_mass;
            return cnt ? (unsigned long long)cnt * wfix(K::value_of_key(kmax - (uint32_t)d)) : 0ull;
          };
          unsigned long long Z = zrow;
          if (topk_on) {          // Z of the top-k set: its bins all lie in the window
            Z = 0;
            for (int d0 = 0, d1 = 0; d0 <= dk; d0 = d1) {      // dk < covered
              d1 = min(d0 + kWinBlock, covered);
              unsigned int cnt[2];
              row_counts(d0, d1, cnt);
              Z += block_sum_u64(bin_mass(d0 + tid * 2, d1, cnt[0]) + bin_mass(d0 + tid * 2 + 1, d1, cnt[1]), h.red);
            }
          }
          const unsigned long long P = (unsigned long long)((double)p * (double)Z);
          unsigned long long before = 0;
          for (int d0 = 0, d1 = 0; d0 < kWinTop && d0 <= dk && !nucleus_done; d0 = d1) {
            if (d0 >= covered) widen();
            d1 = min(d0 + kWinBlock, covered);
            unsigned int cnt[2];
            row_counts(d0, d1, cnt);
            const unsigned long long mb0 = bin_mass(d0 + tid * 2, d1, cnt[0]), mb1 = bin_mass(d0 + tid * 2 + 1, d1, cnt[1]);
            const unsigned long long mine = mb0 + mb1;
            unsigned long long tot;
            const unsigned long long acc = before + block_excl_scan_u64(mine, h.red, tot);
            if (acc <= P && P < acc + mine) h.sel_aux = d0 + tid * 2 + (acc + mb0 > P ? 0 : 1);
            __syncthreads();
            if (before + tot > P) {
              tau = kmax - (uint32_t)h.sel_aux;
              nucleus_done = true;
            }
            before += tot;
          }
        }
      }
      const float mrow = m;     // the row max (this CTA's own when no window was needed: a safe bound)

      // cuts the window cannot answer: radix selection over the slice.  The
      // bins overlay the windows, so first wait until no peer reads them.
      if (!topk_done) {
        cluster_sync();
        windows_free = true;
        list_ok = false;
        uint32_t prefix = 0;
        unsigned long long remaining = (unsigned long long)k;
        for (int shift = 8; shift >= 0; shift -= 8) {
          for (int i = tid; i < kHistCopies * 256; i += kSampThreads) (&hist[0][0])[i] = 0ull;
          __syncthreads();
          const uint32_t hi_mask = shift == 8 ? 0u : 0xff00u;
          visit<T>(slice_smem, n, true, [&](int, uint32_t b) {
            const uint32_t key = K::key(b);
            if ((key & hi_mask) == (prefix & hi_mask))
              atomicAdd(reinterpret_cast<unsigned int*>(&hist[copy][(key >> shift) & 255u]), 1u);
          });
          __syncthreads();
          if (tid < 256) {
            unsigned long long s2 = 0;
            for (int cp = 0; cp < kHistCopies; ++cp) s2 += (unsigned int)(hist[cp][tid] & 0xffffffffull);
            h.ex_arr[c.ex][tid] = s2;
          }
          cluster_sum_array(c);
          select_bin<true>(h, remaining, false);
          const int bin = h.sel_bin;
          remaining -= h.sel_before;
          prefix |= (uint32_t)bin << shift;
          if (shift == 0) cnt_eq = (long long)h.tot[bin];
          __syncthreads();
        }
        kth = prefix;
        need_eq = (long long)remaining;
        topk_done = true;
      }
      if (!nucleus_done) {
        if (!windows_free) cluster_sync();
        windows_free = true;
        list_ok = false;
        auto wfix = [&](float x) -> unsigned long long { return fixed_weight(exp2f((x - mrow) * l2t)); };
        uint32_t prefix = 0;
        unsigned long long target = 0, above = 0;
        for (int shift = 8; shift >= 0; shift -= 8) {
          for (int i = tid; i < kHistCopies * 256; i += kSampThreads) (&hist[0][0])[i] = 0ull;
          __syncthreads();
          const uint32_t hi_mask = shift == 8 ? 0u : 0xff00u;
          visit<T>(slice_smem, n, true, [&](int, uint32_t b) {
            const uint32_t key = K::key(b);
            if ((key & hi_mask) != (prefix & hi_mask)) return;
            if (topk_on && key <= kth) return;
            atomicAdd(&hist[copy][(key >> shift) & 255u], wfix(K::value(b)));
          });
          __syncthreads();
          if (tid < 256) {
            unsigned long long s2 = 0;
            for (int cp = 0; cp < kHistCopies; ++cp) s2 += hist[cp][tid];
            if (crank == 0 && topk_on && need_eq > 0 && (kth & hi_mask) == (prefix & hi_mask) &&
                (int)((kth >> shift) & 255u) == tid)
              s2 += (unsigned long long)need_eq * wfix(K::value_of_key(kth));
            h.ex_arr[c.ex][tid] = s2;
          }
          cluster_sum_array(c);
          if (shift == 8) target = (unsigned long long)((double)p * (double)sum_tot(h));
          select_bin<true>(h, target - above, true);
          const int bin = h.sel_bin;
          const unsigned long long sb = h.sel_before;
          __syncthreads();
          if (bin < 0) { prefix = 0; break; }
          above += sb;
          prefix |= (uint32_t)bin << shift;
        }
        tau = prefix;
      }

      // ---- F3. this CTA's share of the lowest-index ties at the k-th key
      // (slices are ordered by index, so lower ranks take theirs first), and
      // the index of the last tie it keeps.
      int tie_lim = 0x7fffffff;
      int tie_cand = 0x7fffffff;   // index of this CTA's last kept tie, for the extras (INT_MAX: all kept)
      if (topk_on && need_eq < cnt_eq) {
        const bool hi_ok = kth < 0xffffu;
        const T2 ge_k = key_threshold2<T>(kth), ge_k1 = key_threshold2<T>(hi_ok ? kth + 1u : kth);
        auto tie_bits = [&](const uint4 u) -> uint32_t {
          return pass_bits<T>(u, ge_k) & (hi_ok ? ~pass_bits<T>(u, ge_k1) : 0xffu);
        };
        unsigned long long mine;
        long long before = 0;
        if (!windows_free) {
          // The k-th key came from the window walk, so every rank's window
          // bins still hold its exact count of that key (rank r's bin for
          // row distance d is d - gap[r]): this CTA's ties and those of the
          // lower ranks are read there, with no pass over the slice and no
          // exchange.  Nothing below writes the window, so peers may go on
          // reading it.
          if (warp == 0) {                    // lane r reads rank r's bin (r <= this rank)
            const int d = (int)(kmax - kth);
            const int dr = lane <= (int)crank ? d - h.gap[lane] : -1;
            unsigned int cnt_r = 0u;
            if (dr >= 0) cnt_r = lane == (int)crank ? win[dr] : dsmem_ld_u32(dsmem_addr(&win[dr], (uint32_t)lane));
            unsigned long long b = lane < (int)crank ? cnt_r : 0u;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(FULL_MASK, b, o);
            const unsigned int own = __shfl_sync(FULL_MASK, cnt_r, (int)crank);
            if (lane == 0) {
              h.tie_mine = own;
              h.tie_before = (long long)b;
            }
          }
          __syncthreads();
          mine = h.tie_mine;
          before = h.tie_before;
        } else {
          // the k-th key came from the radix selection (the window is gone):
          // count the ties and exchange the counts
          int tn = 0;
          for (int v = tid; v < nvec; v += kSampThreads) tn += __popc(tie_bits(sv[v]));
          for (int j = rest + tid; j < n; j += kSampThreads) tn += K::key(bits_at(j)) == kth;
          mine = block_sum_u64((unsigned long long)tn, h.red);
          const ulonglong2* px = cluster_push(c, crank, mine, 0ull);
          for (int r = 0; r < (int)crank; ++r) before += (long long)px[r].x;
        }
        const long long want = min(max(need_eq - before, 0ll), (long long)mine);
        if (want == 0) {
          tie_lim = -1;
        } else if (want < (long long)mine) {
          // The want-th tie in index order: each thread counts the ties in a
          // contiguous run of words (the ids past the last word go to the
          // last thread), a block scan places the runs, and the one thread
          // whose run holds the want-th tie walks it to that id.
          const int per = (nvec + kSampThreads - 1) / kSampThreads;
          const int v0 = min(nvec, tid * per), v1 = min(nvec, v0 + per);
          int cnt = 0;
          for (int v = v0; v < v1; ++v) cnt += __popc(tie_bits(sv[v]));
          if (tid == kSampThreads - 1)
            for (int j = rest; j < n; ++j) cnt += K::key(bits_at(j)) == kth;
          if (tid == 0) h.sel_aux = -1;       // ordered before the finder's write by the scan's barriers
          unsigned long long tot_t;
          const long long pos = (long long)block_excl_scan_u64((unsigned long long)cnt, h.red, tot_t);
          if (pos < want && want <= pos + cnt) {
            int r = (int)(want - pos);                    // 1-based rank inside this run
            int at = -1;
            for (int v = v0; v < v1 && at < 0; ++v) {
              uint32_t tb = tie_bits(sv[v]);
              const int c1 = __popc(tb);
              if (r > c1) {
                r -= c1;
                continue;
              }
              for (int q = 1; q < r; ++q) tb &= tb - 1;
              at = v * 8 + __ffs(tb) - 1;
            }
            for (int j = rest; at < 0 && j < n; ++j)       // the last thread's tail ids
              if (K::key(bits_at(j)) == kth && --r == 0) at = j;
            h.sel_aux = at;
          }
          __syncthreads();
          tie_lim = h.sel_aux;
        }
        tie_cand = want == 0 ? -1 : (want == (long long)mine ? lo + n - 1 : lo + tie_lim);
      }

      // ---- F4. Gumbel-max over the kept ids
      uint32_t thr = tau;
      if (topk_on && kth > thr) thr = kth;
      {
        // ids below m - 22 T can never win: fold that into the key threshold
        const float vmin = mrow - 22.f * Tr;
        T tv;
        if constexpr (std::is_same<T, __half>::value) tv = __float2half_rd(vmin);
        else tv = __float2bfloat16_rd(vmin);
        const uint32_t kp = K::key((uint32_t)(*reinterpret_cast<const unsigned short*>(&tv)));
        if (!isinf(vmin) && kp > thr) thr = kp;
      }
      const float invT = 1.f / Tr;
      auto keep = [&](int j, uint32_t b) -> bool {
        const uint32_t key = K::key(b);
        if (key < tau) return false;
        if (topk_on && (key < kth || (key == kth && j > tie_lim))) return false;
        return (K::value(b) - mrow) * invT >= -kGumbelSpan;
      };
      auto score_of = [&](int jg, uint32_t b) -> unsigned long long {
        return race_key(seed, off, (uint32_t)jg, (mrow - K::value(b)) * l2t);
      };
      unsigned long long bestg = 0;
      // The first window's list holds every candidate when the cut lies in
      // the window (thr >= its lowest key); each warp then compacts its
      // own segment of the list in place and scores it.  Otherwise the
      // candidates are compacted from the slice into a CTA-wide list after
      // the full window (count pass, block scan, write pass), in rounds if
      // they do not fit.  Either way Philox and the logarithms run on full
      // warps.
      if (list_ok) {
        const int seg = ((list_n + kSampWarps - 1) / kSampWarps + 31) & ~31;
        const int s0 = min(list_n, warp * seg), s1 = min(list_n, s0 + seg);
        int wpos = s0;
        for (int base = s0; base < s1; base += 32) {
          const int i = base + lane;
          const uint32_t j = i < s1 ? list[i] : 0u;
          const bool pass = i < s1 && K::key(bits_at((int)j)) >= thr;
          const unsigned mask = __ballot_sync(FULL_MASK, pass);
          // every lane loaded before the ballot, and writes land at or
          // below the slots this warp has read
          if (pass) list[wpos + __popc(mask & ((1u << lane) - 1u))] = j;
          wpos += __popc(mask);
        }
        __syncwarp();
        for (int i = s0 + lane; i < wpos; i += 32) {
          const int j = (int)list[i];
          const uint32_t b = bits_at(j);
          if (keep(j, b)) {
            const unsigned long long pk = score_of(lo + j, b);
            bestg = pk > bestg ? pk : bestg;
          }
        }
      } else {
        // the windows are free once no peer walks them; list_ok is
        // cluster-uniform until the windows are free, so this is too
        if (need_win && !windows_free) cluster_sync();
        const int cap = a.list_cap + kWin1;      // every entry of the region
        uint32_t* cl = win;
        const T2 thr_v2 = key_threshold2<T>(thr);
        int mine = 0;
        for (int v = tid; v < nvec; v += kSampThreads) mine += __popc(pass_bits<T>(sv[v], thr_v2));
        for (int j = rest + tid; j < n; j += kSampThreads) mine += K::key(bits_at(j)) >= thr;
        unsigned long long total_u;
        const int first = (int)block_excl_scan_u64((unsigned long long)mine, h.red, total_u);
        const int total = (int)total_u;
        // Dense candidates (sampling close to the plain softmax): more than a
        // quarter of the slice, and more than four per thread (below that one
        // candidate per thread in parallel is quicker): walk the words instead
        // of compacting, one Philox call per group of four ids that holds a
        // candidate (the slice starts on a multiple of 8 ids, so groups never
        // straddle words), the same uniforms per id.
        const bool dense = (long long)total * 4 > (long long)n && total > 4 * kSampThreads;
        if (dense) {
          for (int v = tid; v < nvec; v += kSampThreads) {
            const uint32_t cb = pass_bits<T>(sv[v], thr_v2);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t hb = (cb >> (4 * half)) & 0xfu;
              if (!hb) continue;
              const int j0 = v * 8 + half * 4;
              const uint4 w4 = noise_words(seed, off, (uint32_t)(lo + j0) >> 2);
              const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (!((hb >> e) & 1u)) continue;
                const int j = j0 + e;
                const uint32_t b = bits_at(j);
                if (keep(j, b)) {
                  const unsigned long long pk =
                      race_key_of(noise_of_word(ws[e]), (uint32_t)(lo + j), (mrow - K::value(b)) * l2t);
                  bestg = pk > bestg ? pk : bestg;
                }
              }
            }
          }
          for (int j = rest + tid; j < n; j += kSampThreads) {
            const uint32_t b = bits_at(j);
            if (K::key(b) >= thr && keep(j, b)) {
              const unsigned long long pk = score_of(lo + j, b);
              bestg = pk > bestg ? pk : bestg;
            }
          }
        }
        for (int r0 = 0; !dense && r0 < total; r0 += cap) {   // block-uniform
          const int r1 = min(total, r0 + cap);
          if (mine > 0 && first < r1 && first + mine > r0) {
            int kk = first;                                 // list rank of this thread's next candidate
            for (int v = tid; v < nvec && kk < r1; v += kSampThreads) {
              uint32_t cb = pass_bits<T>(sv[v], thr_v2);
              while (cb) {
                const int e = __ffs(cb) - 1;
                cb &= cb - 1;
                if (kk >= r0 && kk < r1) cl[kk - r0] = (uint32_t)(v * 8 + e);
                ++kk;
              }
            }
            for (int j = rest + tid; j < n && kk < r1; j += kSampThreads) {
              if (K::key(bits_at(j)) < thr) continue;
              if (kk >= r0) cl[kk - r0] = (uint32_t)j;
              ++kk;
            }
          }
          __syncthreads();
          for (int i = tid; i < r1 - r0; i += kSampThreads) {
            const int j = (int)cl[i];
            const uint32_t b = bits_at(j);
            if (keep(j, b)) {
              const unsigned long long pk = score_of(lo + j, b);
              bestg = pk > bestg ? pk : bestg;
            }
          }
          __syncthreads();
        }
      }
      bestg = block_max_u64(bestg, h.red);
      // Race times were taken against this CTA's bound mrow.  When every
      // rank used the same bound (the row max) the packed keys compare as
      // they are; otherwise each rank's best time moves to the row max in
      // log2 units: log2 t + (max - mrow) / (T ln 2).
      const ulonglong2* px = cluster_push(c, crank, bestg,
                                          ((unsigned long long)tie_code(tie_cand) << 32) | __float_as_uint(mrow));
      // warp 0 combines the ranks, lane r taking rank r, and hands the
      // result to the CTA through shared memory (every CTA computes the same
      // answer from the same table, so it is cluster-uniform)
      if (warp == 0) {
        const bool has = lane < c.cs;
        const ulonglong2 pr = has ? px[lane] : make_ulonglong2(0ull, 0ull);
        const float mr_l = __uint_as_float((uint32_t)pr.y);
        float mm_w = has ? mr_l : -INFINITY;
        uint32_t te = has ? (uint32_t)(pr.y >> 32) : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          mm_w = fmaxf(mm_w, __shfl_xor_sync(FULL_MASK, mm_w, o));
          te = max(te, __shfl_xor_sync(FULL_MASK, te, o));
        }
        const bool same = __all_sync(FULL_MASK, !has || (uint32_t)pr.y == (uint32_t)px[0].y);
        unsigned long long bw = has ? pr.x : 0ull;
        if (same) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long t = __shfl_xor_sync(FULL_MASK, bw, o);
            bw = t > bw ? t : bw;
          }
        } else {
          // the smallest log2 race time wins, then the lowest id (the
          // largest low word); ranks without a candidate carry +inf
          float lr = INFINITY;
          if (bw != 0) lr = log2f(Keys<float>::value_of_key(~(uint32_t)(bw >> 32))) + (mm_w - mr_l) * l2t;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float lo2 = __shfl_xor_sync(FULL_MASK, lr, o);
            const unsigned long long bo = __shfl_xor_sync(FULL_MASK, bw, o);
            const bool take = bo != 0 && (bw == 0 || lo2 < lr || (lo2 == lr && (uint32_t)bo > (uint32_t)bw));
            if (take) {
              lr = lo2;
              bw = bo;
            }
          }
        }
        if (lane == 0) {
          h.fin_best = bw;
          h.fin_mm = mm_w;
          h.fin_tie = te;
        }
      }
      __syncthreads();
      unsigned long long best = h.fin_best;
      const uint32_t tie_enc = h.fin_tie;
      const float mm = h.fin_mm;
      // the max allowed id passes every filter, so best is 0 only when no id
      // is allowed (or none is finite)
      const bool uniform = best == 0;
      if (uniform) best = uniform_draw();
      if (crank == 0 && tid == 0) a.token_ids[row_id] = (int)(0xffffffffu - (uint32_t)(best & 0xffffffffull));
      put_row_info((uniform ? kRowUniform : 0) | (topk_on ? kRowTopK : 0), tau, kth, tie_enc, mm);
      return;
    }
  }

  // ---- 0. slice -> shared memory (bulk copies, one barrier per chunk)
  const T* src = row + lo;
  bool vec = a.vec != 0;
  if (a.resident) {
    const int bytes = n * (int)sizeof(T);
    const int bulk = bytes & ~15;
    const int nch = (bulk + kChunkBytes - 1) / kChunkBytes;
    if (tid == 0) {                 // copies issued before the barrier, as in the fast path
      for (int i = 0; i < nch; ++i) mbar_init(&h.bar[i], 1);
      fence_mbar_init();
      for (int i = 0; i < nch; ++i) {
        const int off = i * kChunkBytes;
        const int sz = min(kChunkBytes, bulk - off);
        mbar_arrive_expect_tx(&h.bar[i], (uint32_t)sz);
        bulk_g2s(reinterpret_cast<uint8_t*>(slice_smem) + off, reinterpret_cast<const uint8_t*>(src) + off,
                 (uint32_t)sz, &h.bar[i]);
      }
    }
    __syncthreads();
    for (int j = bulk / (int)sizeof(T) + tid; j < n; j += kSampThreads) slice_smem[j] = src[j];
    for (int i = 0; i < nch; ++i) mbar_wait_bounded(&h.bar[i], 0);
    __syncthreads();
    if (mask_row) {                 // masked ids become -inf in place (masks need a resident slice)
      for (int j = tid; j < n; j += kSampThreads)
        if (!allowed_bit(mask_row, lo + j)) slice_smem[j] = neg_inf_value<T>();
      __syncthreads();
    }
    src = slice_smem;
    vec = true;
  }

  // ---- 1. max key and the lowest index holding it (row-wide)
  unsigned long long best = 0;
  visit<T>(src, n, vec, [&](int j, uint32_t b) {
    const unsigned long long pk = ((unsigned long long)K::key(b) << 32) | (0xffffffffu - (uint32_t)(lo + j));
    best = pk > best ? pk : best;
  });
  best = block_max_u64(best, h.red);
  cluster_wait();                                   // every peer has started
  best = cluster_scalar<true>(c, best);
  const uint32_t kmax = (uint32_t)(best >> 32);
  const int imax = (int)(0xffffffffu - (uint32_t)(best & 0xffffffffu));
  const float Tr = row_T;
  if (!(Tr > 0.f)) {
    if (crank == 0 && tid == 0) a.token_ids[row_id] = imax;
    put_row_info(kRowGreedy, 0u, 0u, 0u, 0.f);
    cluster_sync();               // peers may still read this CTA's shared memory
    return;
  }
  const float m = K::value_of_key(kmax);
  const float l2t = 1.4426950408889634f / Tr;
  auto wfix = [&](float x) -> unsigned long long { return fixed_weight(exp2f((x - m) * l2t)); };

  const int k = row_k;
  const bool topk_on = k > 0 && k < a.V;
  const float p = row_p;
  const bool nucleus_on = p < 1.f;
  uint32_t kth = 0;          // key of the k-th largest
  long long need_eq = 0, cnt_eq = 0;
  uint32_t tau = 0;          // keep key >= tau
  bool topk_done = false, nucleus_done = false;

  // ---- 3. generic top-k: MSB-first radix select with cluster-summed bins
  if (topk_on && !topk_done) {
    uint32_t prefix = 0;
    unsigned long long remaining = (unsigned long long)k;
    for (int shift = KB - 8; shift >= 0; shift -= 8) {
      for (int i = tid; i < kHistCopies * 256; i += kSampThreads) (&hist[0][0])[i] = 0ull;
      __syncthreads();
      const uint32_t hi_mask = (shift + 8 >= 32) ? 0u : (~0u << (shift + 8));
      visit<T>(src, n, vec, [&](int, uint32_t b) {
        const uint32_t key = K::key(b);
        if ((key & hi_mask) == (prefix & hi_mask))
          atomicAdd(reinterpret_cast<unsigned int*>(&hist[copy][(key >> shift) & 255u]), 1u);
      });
      __syncthreads();
      if (tid < 256) {
        unsigned long long s = 0;
        for (int cp = 0; cp < kHistCopies; ++cp) s += (unsigned int)(hist[cp][tid] & 0xffffffffull);
        h.ex_arr[c.ex][tid] = s;
      }
      cluster_sum_array(c);
      select_bin<true>(h, remaining, false);
      const int bin = h.sel_bin;
      remaining -= h.sel_before;
      prefix |= (uint32_t)bin << shift;
      if (shift == 0) cnt_eq = (long long)h.tot[bin];
      __syncthreads();
    }
    kth = prefix;
    need_eq = (long long)remaining;
  }

  // ---- 4. generic nucleus: radix select on cluster-summed fixed-point mass
  if (nucleus_on && !nucleus_done) {
    uint32_t prefix = 0;
    unsigned long long target = 0, above = 0;
    for (int shift = KB - 8; shift >= 0; shift -= 8) {
      for (int i = tid; i < kHistCopies * 256; i += kSampThreads) (&hist[0][0])[i] = 0ull;
      __syncthreads();
      const uint32_t hi_mask = (shift + 8 >= 32) ? 0u : (~0u << (shift + 8));
      visit<T>(src, n, vec, [&](int, uint32_t b) {
        const uint32_t key = K::key(b);
        if ((key & hi_mask) != (prefix & hi_mask)) return;
        if (topk_on && key <= kth) return;     // the k-th key's ties are added below
        atomicAdd(&hist[copy][(key >> shift) & 255u], wfix(K::value(b)));
      });
      __syncthreads();
      if (tid < 256) {
        unsigned long long s = 0;
        for (int cp = 0; cp < kHistCopies; ++cp) s += hist[cp][tid];
        if (crank == 0 && topk_on && need_eq > 0 && (kth & hi_mask) == (prefix & hi_mask) &&
            (int)((kth >> shift) & 255u) == tid)
          s += (unsigned long long)need_eq * wfix(K::value_of_key(kth));
        h.ex_arr[c.ex][tid] = s;
      }
      cluster_sum_array(c);
      if (shift == KB - 8) {
        unsigned long long Z = 0;
        for (int b = 0; b < 256; ++b) Z += h.tot[b];
        target = (unsigned long long)((double)p * (double)Z);
      }
      select_bin<true>(h, target - above, true);
      const int bin = h.sel_bin;
      const unsigned long long sb = h.sel_before;
      __syncthreads();
      if (bin < 0) {            // the whole set is needed to exceed p: keep all
        prefix = 0;
        break;
      }
      above += sb;
      prefix |= (uint32_t)bin << shift;
    }
    tau = prefix;
  }

  // ---- 5. ties at the k-th key straddling the cut: this CTA's share of the
  // lowest-index ties (slices are ordered by index), found by a local radix
  // select over its tie indices; tie_lim = largest local index kept
  int tie_lim = 0x7fffffff;
  int tie_cand = 0x7fffffff;     // index of this CTA's last kept tie, for the extras (INT_MAX: all kept)
  if (topk_on && need_eq < cnt_eq) {
    unsigned long long mine = 0;
    visit<T>(src, n, vec, [&](int, uint32_t b) { mine += K::key(b) == kth; });
    mine = block_sum_u64(mine, h.red);
    long long before = 0;
    {
      const ulonglong2* px = cluster_push(c, crank, mine, 0ull);
      for (int r = 0; r < (int)crank; ++r) before += (long long)px[r].x;
    }
    const long long want = min(max(need_eq - before, 0ll), (long long)mine);
    if (want == 0) {
      tie_lim = -1;
    } else if (want < (long long)mine) {
      uint32_t prefix = 0;
      unsigned long long remaining = (unsigned long long)want;
      for (int shift = 16; shift >= 0; shift -= 8) {
        for (int i = tid; i < kHistCopies * 256; i += kSampThreads) (&hist[0][0])[i] = 0ull;
        __syncthreads();
        const uint32_t hi_mask = (shift + 8 >= 24) ? 0u : ((~0u << (shift + 8)) & 0xffffffu);
        visit<T>(src, n, vec, [&](int j, uint32_t b) {
          if (K::key(b) != kth) return;
          const uint32_t ik = 0xffffffu - (uint32_t)j;
          if ((ik & hi_mask) == (prefix & hi_mask))
            atomicAdd(reinterpret_cast<unsigned int*>(&hist[copy][(ik >> shift) & 255u]), 1u);
        });
        __syncthreads();
        if (tid < 256) {
          unsigned long long s = 0;
          for (int cp = 0; cp < kHistCopies; ++cp) s += (unsigned int)(hist[cp][tid] & 0xffffffffull);
          h.tot[tid] = s;
        }
        __syncthreads();
        select_bin<true>(h, remaining, false);
        remaining -= h.sel_before;
        prefix |= (uint32_t)h.sel_bin << shift;
        __syncthreads();
      }
      tie_lim = (int)(0xffffffu - prefix);
    }
    tie_cand = want == 0 ? -1 : (want == (long long)mine ? lo + n - 1 : lo + tie_lim);
  }

  // ---- 6. Gumbel-max over the kept ids, candidates queued per warp
  const float invT = 1.f / Tr;
  unsigned long long bestg = 0;
  uint32_t* qi = q_idx + warp * kQueue;
  float* qx = q_x + warp * kQueue;
  int qh = 0, qn = 0;
  __syncthreads();                              // the region now holds the queues
  auto keep = [&](int j, uint32_t b) -> bool {
    const uint32_t key = K::key(b);
    if (key < tau) return false;
    if (topk_on && (key < kth || (key == kth && j > tie_lim))) return false;
    return (K::value(b) - m) * invT >= -kGumbelSpan;
  };
  auto drain = [&](int cnt) {
    if (lane < cnt) {
      const int slot = (qh + lane) & (kQueue - 1);
      const uint32_t j = qi[slot];
      const unsigned long long pk = race_key(seed, off, j, (m - qx[slot]) * l2t);
      bestg = pk > bestg ? pk : bestg;
    }
    __syncwarp();
    qh = (qh + cnt) & (kQueue - 1);
    qn -= cnt;
  };
  auto push = [&](bool cand, int j, uint32_t b) {
    const unsigned mask = __ballot_sync(FULL_MASK, cand);
    if (mask) {
      if (cand) {
        const int slot = (qh + qn + __popc(mask & ((1u << lane) - 1u))) & (kQueue - 1);
        qi[slot] = (uint32_t)(lo + j);
        qx[slot] = K::value(b);
      }
      qn += __popc(mask);
      __syncwarp();
      if (qn >= 32) drain(32);
    }
  };
  {
    const int nvec = vec ? n / E : 0;
    const uint4* sv = reinterpret_cast<const uint4*>(src);
    for (int vb = warp * 32; vb < nvec; vb += kSampThreads) {     // warp-uniform trip count
      const int v = vb + lane;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (v < nvec) u = sv[v];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint32_t b = (sizeof(T) == 4) ? w[e] : ((w[e / 2] >> (16 * (e & 1))) & 0xffffu);
        const int j = v * E + e;
        push(v < nvec && keep(j, b), j, b);
      }
    }
    for (int jb = nvec * E + warp * 32; jb < n; jb += kSampThreads) {
      const int j = jb + lane;
      uint32_t b = 0;
      if (j < n)
        b = sizeof(T) == 4 ? __float_as_uint(*reinterpret_cast<const float*>(src + j))
                           : (uint32_t)(*reinterpret_cast<const unsigned short*>(src + j));
      push(j < n && keep(j, b), j, b);
    }
    if (qn > 0) drain(qn);
  }
  bestg = block_max_u64(bestg, h.red);
  uint32_t tie_enc = 0;
  {
    const ulonglong2* px = cluster_push(c, crank, bestg, (unsigned long long)tie_code(tie_cand));
    bestg = 0;
    for (int r = 0; r < c.cs; ++r) {
      bestg = px[r].x > bestg ? px[r].x : bestg;
      tie_enc = max(tie_enc, (uint32_t)px[r].y);
    }
  }
  // 0 only when no id is allowed (or none is finite): uniform over the row
  const bool uniform = bestg == 0;
  if (uniform) bestg = uniform_draw();
  if (crank == 0 && tid == 0) a.token_ids[row_id] = (int)(0xffffffffu - (uint32_t)(bestg & 0xffffffffull));
  put_row_info((uniform ? kRowUniform : 0) | (topk_on ? kRowTopK : 0), tau, kth, tie_enc, m);
  cluster_sync();               // peers may still read this CTA's shared memory
}


// Clusters of `cs` CTAs with `smem` bytes each that the GPU runs at once,
// memoised per device and cluster size as one word (smem << 24 | count), so
// concurrent first calls never pair one call's count with another's size.
// A failed query falls back to an SM-count estimate.
template <typename T>
struct ClusterMemo {
  static PerDeviceMemo<uint64_t> by_size[4];
};
template <typename T>
PerDeviceMemo<uint64_t> ClusterMemo<T>::by_size[4];

template <typename T>
static int max_active_clusters(int cs, size_t smem, int sms) {
  const int li = cs == 1 ? 0 : cs == 2 ? 1 : cs == 4 ? 2 : 3;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const uint64_t known = ClusterMemo<T>::by_size[li].get(dev);
  if (known != 0 && (known >> 24) == (uint64_t)smem) return (int)(known & 0xffffff);
  int n = 0;
  if (cudaFuncSetAttribute(sample_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs);
    cfg.blockDim = dim3(kSampThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, sample_kernel<T>, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  if (n <= 0) n = sms / cs > 0 ? sms / cs : 1;
  if (n > 0xffffff) n = 0xffffff;
  ClusterMemo<T>::by_size[li].put(dev, ((uint64_t)smem << 24) | (uint64_t)n);
  return n;
}

template <typename T>
static cudaError_t launch_sample_t(const SampArgs& base, int num_rows, cudaStream_t stream, int* waves_only) {
  constexpr int kMaxSmem = kSampSmem;
  const size_t hdr = ((sizeof(SampHdr) + 127) / 128) * 128;
  const size_t region = (size_t)region_bytes<T>();
  const int esz = (int)sizeof(T);
  const int align = 16 / esz;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // cluster size: for CS in 1, 2, 4, 8 whose slice fits on chip, estimate
  // the time as (waves of clusters the GPU co-schedules) x (ids per CTA)
  // and keep the cheapest, preferring the smaller cluster on a tie
  auto slice_of = [&](int c) { return ((base.V + c - 1) / c + align - 1) / align * align; };
  auto al128 = [](size_t b) { return (b + 127) / 128 * 128; };
  const size_t budget = kMaxSmem - hdr - region;
  const size_t chunk_cap = (size_t)kMaxChunks * kChunkBytes;
  const size_t cap = budget < chunk_cap ? budget : chunk_cap;
  // shared memory of a launch with cluster size c: the windowed 16-bit path
  // takes all of it (the rest of the region holds candidate lists), the
  // others header + slice + region
  auto smem_of = [&](int c, bool res) -> size_t {
    if (res && esz == 2) return (size_t)kMaxSmem;
    return hdr + (res ? al128((size_t)slice_of(c) * esz) : 0) + region;
  };
  int cs = 0;
  long long best_cost = 0;
  for (int c = 1; c <= kMaxCluster; c *= 2) {
    const size_t sb = al128((size_t)slice_of(c) * esz);
    const bool res = base.vec && sb <= cap;
    if (!res && c < kMaxCluster) continue;
    const int act = max_active_clusters<T>(c, smem_of(c, res), sms);
    const long long waves = ((long long)num_rows + act - 1) / act;
    const long long cost = waves * slice_of(c);
    if (cs == 0 || cost < best_cost) {
      cs = c;
      best_cost = cost;
    }
  }
  if (waves_only) {                 // report the waves of the chosen clusters only
    const int act = max_active_clusters<T>(cs, smem_of(cs, base.vec && al128((size_t)slice_of(cs) * esz) <= cap), sms);
    *waves_only = (num_rows + act - 1) / act;
    return cudaSuccess;
  }
  SampArgs a = base;
  a.slice = slice_of(cs);
  const size_t sbytes = al128((size_t)a.slice * esz);
  a.resident = (a.vec && sbytes <= cap) ? 1 : 0;
  a.fast = (esz == 2 && a.resident) ? 1 : 0;
  const size_t smem = smem_of(cs, a.resident != 0);
  a.list_cap = a.fast ? (int)((smem - hdr - sbytes) / 4) - win1_bins<T>() : 0;
  {
    cudaError_t e = cudaFuncSetAttribute(sample_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_rows * cs));
  cfg.blockDim = dim3(kSampThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, sample_kernel<T>, a);
}


// ------------------------------------------------------------ this build's entry points
static SampArgs args_of(const SampleCall& c) {
  const int esz = c.dtype == PKVD_F32 ? 4 : 2;
  SampArgs a;
  a.fast = 0;
  a.list_cap = 0;
  a.token_ids = c.token_ids;
  a.logits = c.logits;
  a.V = c.vocab;
  a.row_stride = c.row_stride;
  a.slice = c.vocab;
  a.resident = 0;
  a.vec = ((reinterpret_cast<uintptr_t>(c.logits) % 16 == 0) && ((c.row_stride * esz) % 16 == 0)) ? 1 : 0;
  a.temperature = c.temperature;
  a.top_k = c.top_k;
  a.top_p = c.top_p;
  a.seeds = c.seeds;
  a.offsets = c.offsets;
  a.mask = c.mask;
  a.mask_stride = c.mask_stride;
  a.row_info = c.row_info;
  return a;
}

cudaError_t sample_launch(const SampleCall& c, cudaStream_t stream, int* waves_only) {
  const SampArgs a = args_of(c);
  if (c.dtype == PKVD_F32) return launch_sample_t<float>(a, c.num_rows, stream, waves_only);
  if (c.dtype == PKVD_F16) return launch_sample_t<__half>(a, c.num_rows, stream, waves_only);
  return launch_sample_t<__nv_bfloat16>(a, c.num_rows, stream, waves_only);
}

bool sample_mask_fits(int dtype, int vocab, int64_t row_stride, const void* logits) {
  // a mask is applied to the shared-memory copy of the row: rows must be
  // 16-byte aligned and fit on chip over a cluster of kMaxCluster CTAs
  const int esz = dtype == PKVD_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(logits) % 16) || ((row_stride * esz) % 16)) return false;
  const size_t hdr = ((sizeof(SampHdr) + 127) / 128) * 128;
  const size_t region = esz == 4 ? (size_t)region_bytes<float>() : (size_t)region_bytes<__half>();
  const int align = 16 / esz;
  const long long slice = (((long long)vocab + kMaxCluster - 1) / kMaxCluster + align - 1) / align * align;
  const size_t sb = ((size_t)slice * esz + 127) / 128 * 128;
  const size_t budget = kSampSmem - hdr - region;
  const size_t cap = budget < (size_t)kMaxChunks * kChunkBytes ? budget : (size_t)kMaxChunks * kChunkBytes;
  return sb <= cap;
}

}  // namespace PKVD_SAMP_NS
}  // namespace pkvd
