// The sampler's entry points: the kernel built with 1024-thread CTAs (one per
// SM), the extras kernel, and the choice between this build and the
// 512-thread one (sampler512.cu, two CTAs per SM) for each launch.
#define PKVD_SAMP_THREADS 1024
#define PKVD_SAMP_NS s1024
#include "sampler_core.cuh"

namespace pkvd {
using namespace s1024;   // the helpers the extras kernel shares with the sampler

// ---------------------------------------------------------------- extras
// token_prob and the top-8 of the distribution the draw used (Grok-1
// "第 8 章 runners.py 推理引擎", section 8.3 sample_token and section 8.3.2
// TOP_K = 8): probabilities are softmax of the filtered logits, kept ids as
// they are and every other id at probability 0; the top-8 lists the kept
// ids by value (index order among equal values), then the ids of
// probability 0 in index order.  A cluster of 8 CTAs per row runs after the
// sampler, which left the row's cut parameters (row_info: cut keys, the last
// kept tie at the k-th key, the row max) and token; each CTA takes one slice
// in one coalesced pass and pushes its partials to rank 0.
struct ExtrasArgs {
  const void* logits;
  int V;
  int64_t row_stride;
  const float* temperature;
  const uint32_t* mask;
  int64_t mask_stride;
  const int32_t* row_info;
  const int32_t* token_ids;
  float* token_prob;      // [rows] or null
  float* top_probs;       // [rows, 8] or null
  int32_t* top_ids;       // [rows, 8] or null
};

constexpr int kTop = 8;
constexpr int kExThreads = 512;            // threads per extras CTA
constexpr int kExCluster = 8;              // CTAs (slices) per row
constexpr int kExWarps = kExThreads / 32;

// 8 rounds of a warp-wide max over the heads of per-lane lists sorted in
// descending order; the owner of each winner pops it (entries are unique).
__device__ __forceinline__ void warp_merge8(unsigned long long* lst, unsigned long long* outl) {
#pragma unroll
  for (int i = 0; i < kTop; ++i) {
    unsigned long long best = lst[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(FULL_MASK, best, o));
    outl[i] = best;
    if (best != 0ull && lst[0] == best) {
#pragma unroll
      for (int q = 0; q < kTop - 1; ++q) lst[q] = lst[q + 1];
      lst[kTop - 1] = 0ull;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kExThreads) sample_extras_kernel(const ExtrasArgs e) {
  using K = Keys<T>;
  // per-rank partials pushed to rank 0: [rank][0] Z (f64 bits), [1] kept
  // count, [2..9] the rank's best 8 (key, -index)
  __shared__ unsigned long long s_part[kExCluster][2 + kTop];
  __shared__ unsigned long long s_top[kExWarps][kTop];
  __shared__ double s_z[kExWarps];
  __shared__ long long s_n[kExWarps];
  pdl_wait();                       // the sampler's token and row_info
  pdl_trigger();
  cluster_arrive_relaxed();         // matched by cluster_wait() before the push to rank 0
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const int r = blockIdx.x / kExCluster;
  const T* row = static_cast<const T*>(e.logits) + (int64_t)r * e.row_stride;
  const uint32_t* mrow = e.mask ? e.mask + (int64_t)r * e.mask_stride : nullptr;
  const int32_t* info = e.row_info + (int64_t)r * kRowInfo;
  const int flags = info[0];
  const int tok = e.token_ids[r];
  const int V = e.V;
  auto bits_of = [&](int j) -> uint32_t {
    if constexpr (sizeof(T) == 4) return __float_as_uint(reinterpret_cast<const float*>(row)[j]);
    else return (uint32_t)reinterpret_cast<const unsigned short*>(row)[j];
  };
  auto allowed = [&](int j) { return !mrow || allowed_bit(mrow, j); };
  float* tp = e.top_probs ? e.top_probs + (int64_t)r * kTop : nullptr;
  int32_t* ti = e.top_ids ? e.top_ids + (int64_t)r * kTop : nullptr;
  if (flags & (kRowGreedy | kRowUniform)) {
    // a point mass on the token, or every id equal (nothing allowed); the
    // branch is the same on every rank, so no rank waits at a barrier
    if (crank == 0 && tid == 0) {
      const bool uni = (flags & kRowUniform) != 0;
      const float pu = 1.f / (float)V;
      if (e.token_prob) e.token_prob[r] = uni ? pu : 1.f;
      int fill = 0, next = 0;
      if (!uni) {
        if (tp) tp[0] = 1.f;
        if (ti) ti[0] = tok;
        fill = 1;
      }
      for (; fill < kTop; ++fill) {
        if (!uni && next == tok) ++next;
        const bool in = next < V;
        if (tp) tp[fill] = in ? (uni ? pu : 0.f) : 0.f;
        if (ti) ti[fill] = in ? next : -1;
        ++next;
      }
    }
    cluster_wait();
    return;
  }
  const float Tr = e.temperature[r];
  const float l2t = 1.4426950408889634f / Tr;
  const bool topk = (flags & kRowTopK) != 0;
  const uint32_t tau = (uint32_t)info[1], kth = (uint32_t)info[2];
  const int tie_last = info[3];
  const float m = __int_as_float(info[4]);
  const uint32_t thr = topk && kth > tau ? kth : tau;
  // kept: allowed, at or above the cut, and at the k-th key only up to the
  // last kept tie (the sampler keeps the lowest indices)
  auto kept = [&](int j, uint32_t key) {
    return allowed(j) && key >= thr && !(topk && key == kth && j > tie_last);
  };
  // this rank's slice of the row, in 16-byte words when the row is aligned
  constexpr int E = 16 / (int)sizeof(T);
  const int per = ((V + kExCluster - 1) / kExCluster + E - 1) / E * E;
  const int lo = min(V, (int)crank * per), hi = min(V, lo + per);
  float zs = 0.f, zc = 0.f;
  unsigned long long t8[kTop];
#pragma unroll
  for (int i = 0; i < kTop; ++i) t8[i] = 0ull;
  int npos = 0;
  auto zadd = [&](float w) {
    const float y = w - zc;
    const float t = zs + y;
    zc = (t - zs) - y;
    zs = t;
  };
  auto insert = [&](unsigned long long pk) {
    if (pk > t8[kTop - 1]) {
      t8[kTop - 1] = pk;
#pragma unroll
      for (int i = kTop - 1; i > 0; --i)
        if (t8[i] > t8[i - 1]) {
          const unsigned long long x = t8[i];
          t8[i] = t8[i - 1];
          t8[i - 1] = x;
        }
    }
  };
  auto take = [&](int j, uint32_t b) {
    const uint32_t key = K::key(b);
    if (!kept(j, key)) return;
    ++npos;
    zadd(ex2_ftz((K::value(b) - m) * l2t));
    insert(((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)j));
  };
  const bool vec = (reinterpret_cast<uintptr_t>(row) % 16) == 0;
  const int nvec = vec ? (hi - lo) / E : 0;
  const uint4* rv = reinterpret_cast<const uint4*>(row + lo);
  if constexpr (sizeof(T) == 2) {
    // a packed compare against the cut finds the few words with kept ids
    const auto thr2 = key_threshold2<T>(thr);
    const bool plain = !mrow && !topk;          // kept == at or above the cut
    for (int v = tid; v < nvec; v += kExThreads) {
      const uint4 u = rv[v];
      uint32_t pb = pass_bits<T>(u, thr2);
      if (plain && pb == 0xffu) {
        // a whole word kept: its 8 weights summed as a tree, one compensated
        // add, and the keys tested against this thread's 8th best
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        const float ml = m * l2t;
        float ws = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = Pack2<T>::to_float2(w[q]);
          ws += ex2_ftz(fmaf(f.x, l2t, -ml)) + ex2_ftz(fmaf(f.y, l2t, -ml));
        }
        zadd(ws);
        npos += 8;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t b = (w[q / 2] >> (16 * (q & 1))) & 0xffffu;
          insert(((unsigned long long)K::key(b) << 32) | (0xffffffffu - (uint32_t)(lo + v * E + q)));
        }
        continue;
      }
      while (pb) {
        const int q = __ffs(pb) - 1;
        pb &= pb - 1;
        const uint32_t wd = q < 2 ? u.x : (q < 4 ? u.y : (q < 6 ? u.z : u.w));
        take(lo + v * E + q, (q & 1) ? (wd >> 16) : (wd & 0xffffu));
      }
    }
  } else {
    for (int v = tid; v < nvec; v += kExThreads) {
      const uint4 u = rv[v];
      take(lo + v * 4 + 0, u.x);
      take(lo + v * 4 + 1, u.y);
      take(lo + v * 4 + 2, u.z);
      take(lo + v * 4 + 3, u.w);
    }
  }
  for (int j = lo + nvec * E + tid; j < hi; j += kExThreads) take(j, bits_of(j));
  // block: Z, the kept count, the best 8
  double z = (double)zs;
  long long np = npos;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    z += __shfl_xor_sync(FULL_MASK, z, o);
    np += __shfl_xor_sync(FULL_MASK, np, o);
  }
  unsigned long long wl[kTop];
  warp_merge8(t8, wl);
  if (lane == 0) {
    s_z[warp] = z;
    s_n[warp] = np;
#pragma unroll
    for (int i = 0; i < kTop; ++i) s_top[warp][i] = wl[i];
  }
  __syncthreads();
  cluster_wait();                   // every rank has started: rank 0's table may be written
  if (warp == 0) {
    double zb = lane < kExWarps ? s_z[lane] : 0.0;
    long long nb = lane < kExWarps ? s_n[lane] : 0;
    unsigned long long ll[kTop], bl[kTop];
#pragma unroll
    for (int i = 0; i < kTop; ++i) ll[i] = lane < kExWarps ? s_top[lane][i] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      zb += __shfl_xor_sync(FULL_MASK, zb, o);
      nb += __shfl_xor_sync(FULL_MASK, nb, o);
    }
    warp_merge8(ll, bl);
    // push this rank's partials into rank 0's table
    if (lane < 2 + kTop) {
      const unsigned long long val = lane == 0 ? (unsigned long long)__double_as_longlong(zb)
                                   : lane == 1 ? (unsigned long long)nb : bl[0];
      unsigned long long vv = val;
#pragma unroll
      for (int i = 0; i < kTop; ++i)
        if (lane == 2 + i) vv = bl[i];
      const uint32_t addr = dsmem_addr(&s_part[crank][lane], 0u);
      asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(vv) : "memory");
    }
  }
  cluster_sync();
  if (crank != 0 || warp != 0) return;
  // rank 0: the row's Z, count and best 8 over the ranks
  double Z = lane < kExCluster ? __longlong_as_double((long long)s_part[lane][0]) : 0.0;
  long long NP = lane < kExCluster ? (long long)s_part[lane][1] : 0;
  unsigned long long ll[kTop], fl[kTop];
#pragma unroll
  for (int i = 0; i < kTop; ++i) ll[i] = lane < kExCluster ? s_part[lane][2 + i] : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Z += __shfl_xor_sync(FULL_MASK, Z, o);
    NP += __shfl_xor_sync(FULL_MASK, NP, o);
  }
  warp_merge8(ll, fl);
  if (lane != 0) return;
  const float inv = (float)(1.0 / Z);
  if (e.token_prob) e.token_prob[r] = ex2_ftz((K::value(bits_of(tok)) - m) * l2t) * inv;
  int fill = 0;
  for (; fill < kTop && fl[fill] != 0ull; ++fill) {
    const uint32_t key = (uint32_t)(fl[fill] >> 32);
    if (tp) tp[fill] = ex2_ftz((K::value_of_key(key) - m) * l2t) * inv;
    if (ti) ti[fill] = (int32_t)(0xffffffffu - (uint32_t)(fl[fill] & 0xffffffffull));
  }
  // fewer than 8 kept: the lowest ids of probability 0, in index order
  for (int j = 0; fill < kTop && j < V; ++j) {
    if (kept(j, K::key(bits_of(j)))) continue;
    if (tp) tp[fill] = 0.f;
    if (ti) ti[fill] = j;
    ++fill;
  }
  for (; fill < kTop; ++fill) {
    if (tp) tp[fill] = 0.f;
    if (ti) ti[fill] = -1;
  }
  (void)NP;
}


cudaError_t launch_sample(int32_t* token_ids, const void* logits, int dtype, int num_rows, int vocab,
                          int64_t row_stride, const float* temperature, const int32_t* top_k,
                          const float* top_p, const uint64_t* seeds, const uint64_t* offsets,
                          const uint32_t* mask, int64_t mask_stride, int32_t* row_info, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  const SampleCall c{token_ids, logits, dtype, num_rows, vocab, row_stride, temperature, top_k, top_p, seeds,
                     offsets, mask, mask_stride, row_info};
  // One CTA of 1024 threads per SM while one wave of its clusters covers the
  // rows; when the rows need several waves, two CTAs of 512 threads per SM,
  // so that one computes while the other waits at a barrier or on a peer
  // (measured: 256 rows of 128256 bf16 logits 104.5 -> ~94 us; single-wave
  // batches are no faster and some steps slower that way).
  int waves = 1;
  cudaError_t e = s1024::sample_launch(c, stream, &waves);
  if (e != cudaSuccess) return e;
  const bool split = waves > 1 && (!mask || s512::sample_mask_fits(dtype, vocab, row_stride, logits));
  e = split ? s512::sample_launch(c, stream, nullptr) : s1024::sample_launch(c, stream, nullptr);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool sample_mask_supported(int dtype, int vocab, int64_t row_stride, const void* logits) {
  // the larger build can take every row the smaller one can
  return s1024::sample_mask_fits(dtype, vocab, row_stride, logits);
}

cudaError_t launch_sample_extras(const void* logits, int dtype, int num_rows, int vocab, int64_t row_stride,
                                 const float* temperature, const uint32_t* mask, int64_t mask_stride,
                                 const int32_t* row_info, const int32_t* token_ids, float* token_prob,
                                 float* top_probs, int32_t* top_ids, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  ExtrasArgs x;
  x.logits = logits;
  x.V = vocab;
  x.row_stride = row_stride;
  x.temperature = temperature;
  x.mask = mask;
  x.mask_stride = mask_stride;
  x.row_info = row_info;
  x.token_ids = token_ids;
  x.token_prob = token_prob;
  x.top_probs = top_probs;
  x.top_ids = top_ids;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_rows * kExCluster));
  cfg.blockDim = dim3(kExThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)kExCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (dtype == PKVD_F32) return cudaLaunchKernelEx(&cfg, sample_extras_kernel<float>, x);
  if (dtype == PKVD_F16) return cudaLaunchKernelEx(&cfg, sample_extras_kernel<__half>, x);
  return cudaLaunchKernelEx(&cfg, sample_extras_kernel<__nv_bfloat16>, x);
}

}  // namespace pkvd
