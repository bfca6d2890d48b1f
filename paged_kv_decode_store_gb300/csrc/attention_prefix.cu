// Paged decode attention for a batch whose rows share a cached prefix.
//
// What is computed is the plain decode attention (nano-vllm "Model Runner",
// "prefill and decode"; Grok-1 "第 8 章 runners.py 推理引擎", sections 8.2.3
// and 8.5): for row i, query head h, kv head hk = h / G,
//   out[i,h] = sum_{j < ctx_i} softmax_j(scale * <q[i,h], K_j>) V_j .
// The batch shape is nanochat's ("04 · Engine 推理与工具调用", sections 2-3):
// one prefill is cloned N ways, so the first prefix_len tokens of every row
// are the same cached blocks (every row's first prefix_len / block_size table
// entries name the same physical blocks).  The plain kernel reads those
// blocks once per row; here each is read once per group of rows:
//
// * The work is split in two.  Prefix CTAs each take a sub-group of up to
//   16 / G rows and a contiguous range of the prefix's 16-token chunks; their
//   consumer warps (one per KV head) apply every query of the sub-group (at
//   most 16: two mma n-tiles of 8 queries) to each staged K/V tile, keeping
//   one online-softmax state per query.  Suffix CTAs take an equal stream-K
//   slice of the rows' own chunks after the prefix.
// * Every CTA derives the same plan from the context lengths: the prefix
//   gets CTAs in proportion to its share of the chunk loads (at most 24
//   splits per sub-group, so a row's records load in one round of the
//   merge), the suffix the rest.
// * Nothing is normalised in the partition kernel: every segment leaves an
//   (m, l, acc) record, and the merge kernel (a programmatic dependent)
//   combines a row's prefix records and suffix records with the log-sum-exp
//   identity.
// The producer, stage ring, bounded waits and error flags are the plain
// kernel's (attention_kernels.cuh).
#include "attention_kernels.cuh"

namespace pkvd {

namespace {

constexpr int kPrefixMaxSplits = 24;   // record slots per sub-group (a row's records load in one round)
constexpr int kPrefixQueries = 16;     // queries a consumer warp carries (two n-tiles of 8)

struct PrefixParams {
  PartParams p;          // the call (rec unused)
  int prefix_len;        // shared tokens, a multiple of 16 and of the block size
  int sg_rows;           // rows per sub-group
  int nsg;               // sub-groups
  int max_splits;        // record slots per sub-group (<= kPrefixMaxSplits, <= prefix chunks)
  float* rec;            // records [prefix | suffix CTAs x 2 | rows][hq][D + 4]
  int64_t rec_suffix;    // first suffix-CTA record
  int64_t rec_rows;      // first per-row record
};

struct PrefixPlan {
  int pc;                // prefix chunks
  int splits;            // prefix CTAs per sub-group
  int gp;                // prefix CTAs (nsg * splits)
  int gs;                // suffix CTAs
};

// The plan every CTA (and the merge kernel) derives from the suffix chunk
// total cs.  The host guarantees nsg < grid, so gs >= 1.
__device__ __forceinline__ PrefixPlan prefix_plan(const PrefixParams& q, long long cs, int grid) {
  PrefixPlan pl;
  pl.pc = q.prefix_len / kChunk;
  const long long pref = (long long)q.nsg * pl.pc;
  const long long w = pref + cs;
  const long long target = w > 0 ? (grid * pref + w / 2) / w : 1;      // prefix CTAs by share of loads
  int splits = (int)(target / q.nsg);
  splits = splits < 1 ? 1 : splits;
  splits = splits > q.max_splits ? q.max_splits : splits;
  while (splits > 1 && q.nsg * splits > grid - 1) --splits;
  pl.splits = splits;
  pl.gp = q.nsg * splits;
  pl.gs = grid - pl.gp;
  return pl;
}

// Suffix chunks of row i (the chunks after the shared prefix; 0 for a row
// whose context does not reach past it).
__device__ __forceinline__ int suffix_chunks(const PartParams& p, int i, int pc) {
  const int n = chunks_of(p.ctx, i, p.ctx_cap, 0) - pc;
  return n > 0 ? n : 0;
}

// One consumer warp: KV head hk for up to 16 queries (rows r0 .. r0 + rows - 1,
// G query heads each), online softmax per query, O^T accumulated with
// mma.m16n8k16 in two n-tiles.
template <typename T, int D>
struct GroupConsumer {
  static constexpr int KS = D / 16;
  uint32_t qf[2][KS][2];
  float acc[2][KS][4];
  float m[2][2], l[2][2];
  int r0, nq;

  __device__ void begin(const PartParams& p, int row0, int rows, int warp, int lane) {
    const int lr = lane >> 2, lc = lane & 3;
    r0 = row0;
    nq = rows * p.G;
    const T* qb = static_cast<const T*>(p.q);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int qi = t * 8 + lr;
      const bool ok = qi < nq;
      const int row = ok ? row0 + qi / p.G : row0, g = ok ? qi % p.G : 0;
      const T* src = qb + ((int64_t)row * p.hq + warp * p.G + g) * D;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qf[t][kk][0] = ok ? *reinterpret_cast<const uint32_t*>(src + kk * 16 + 2 * lc) : 0u;
        qf[t][kk][1] = ok ? *reinterpret_cast<const uint32_t*>(src + kk * 16 + 8 + 2 * lc) : 0u;
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[t][kk][r] = 0.f;
      }
      m[t][0] = m[t][1] = -INFINITY;
      l[t][0] = l[t][1] = 0.f;
    }
  }

  __device__ void chunk(const PartParams& p, uint8_t* sK, uint8_t* sV, int ntok, int warp, int lane) {
    constexpr int ESZ = sizeof(T);
    const int lr = lane >> 2;
    const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int a_col = (lane >> 4) * 16;
    const int v_mat = lane >> 3;
    const int v_row = (lane & 7) + (v_mat >> 1) * 8;
    const int v_col = (v_mat & 1) * 8 * ESZ;
    const int hoff = warp * D * ESZ;
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
    // S^T = K Q^T for both n-tiles from one ldmatrix of K per k-step
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint32_t kaddr = smem_u32(sK) + a_row * p.rowb + hoff + a_col;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t a[4];
      ldsm_x4(kaddr + kk * 32, a[0], a[1], a[2], a[3]);
      Mma<T>::run(s[0], a, qf[0][kk][0], qf[0][kk][1]);
      Mma<T>::run(s[1], a, qf[1][kk][0], qf[1][kk][1]);
    }
    const float sl = p.scale_log2;
    uint32_t b0[2], b1[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      // fragment: s0,s1 -> token lr, queries 2lc,2lc+1 ; s2,s3 -> token lr+8
      const float x0 = lr < ntok ? s[t][0] * sl : -INFINITY;
      const float x1 = lr < ntok ? s[t][1] * sl : -INFINITY;
      const float x2 = lr + 8 < ntok ? s[t][2] * sl : -INFINITY;
      const float x3 = lr + 8 < ntok ? s[t][3] * sl : -INFINITY;
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, o));
      }
      const float mn0 = fmaxf(m[t][0], mx0), mn1 = fmaxf(m[t][1], mx1);
      const float c0 = exp2f(m[t][0] - mn0), c1 = exp2f(m[t][1] - mn1);
      const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
      const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
      l[t][0] = l[t][0] * c0 + p0 + p2;
      l[t][1] = l[t][1] * c1 + p1 + p3;
      m[t][0] = mn0;
      m[t][1] = mn1;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        acc[t][mt][0] *= c0;
        acc[t][mt][1] *= c1;
        acc[t][mt][2] *= c0;
        acc[t][mt][3] *= c1;
      }
      b0[t] = movmatrix_trans(Mma<T>::pack(p0, p1));
      b1[t] = movmatrix_trans(Mma<T>::pack(p2, p3));
    }
    // O^T += V^T P^T: one ldmatrix of V^T per m-tile feeds both n-tiles
    const uint32_t vaddr = smem_u32(sV) + v_row * p.rowb + hoff + v_col;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a[4];
      ldsm_x4_trans(vaddr + mt * 16 * ESZ, a[0], a[1], a[2], a[3]);
      Mma<T>::run(acc[0][mt], a, b0[0], b1[0]);
      Mma<T>::run(acc[1][mt], a, b0[1], b1[1]);
    }
  }

  // The unnormalised state of every query into its record: query qi of the
  // segment goes to record rec_first + qi / G (one record per row), head
  // warp * G + qi % G.
  __device__ void finish(const PartParams& p, float* rec, int64_t rec_first, int warp, int lane) {
    const int lr = lane >> 2, lc = lane & 3;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      float lA = l[t][0], lB = l[t][1];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        lA += __shfl_xor_sync(FULL_MASK, lA, o);
        lB += __shfl_xor_sync(FULL_MASK, lB, o);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int qi = t * 8 + 2 * lc + e;
        if (qi >= nq) continue;
        const int h = warp * p.G + qi % p.G;
        float* r = rec + ((rec_first + qi / p.G) * p.hq + h) * (D + 4);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d0 = mt * 16 + lr;
          r[d0] = acc[t][mt][e];
          r[d0 + 8] = acc[t][mt][2 + e];
        }
        if (lr == 0) {
          r[D] = m[t][e];
          r[D + 1] = e ? lB : lA;
        }
      }
    }
  }
};

// meta of a stage: x = first row, y = rows (prefix) or 1, z = tokens | flags << 8,
// w = record index of the segment's first row
enum : int { PF_FIRST = 1, PF_LAST = 2 };

template <typename T, int D>
__global__ void __launch_bounds__(kAttnThreads, 1) paged_decode_prefix_kernel(const PrefixParams q) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const PartParams& p = q.p;
  SmemHdr& hdr = *reinterpret_cast<SmemHdr*>(smem_raw);
  uint8_t* stage_base = smem_raw + ((sizeof(SmemHdr) + 127) / 128) * 128;
  const int stage_bytes = 2 * kChunk * p.rowb;
  const int S = p.stages;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, grid = gridDim.x;
  const int pc = q.prefix_len / kChunk;

  // ---- suffix chunk total (every CTA; CTA 0 flags contexts that do not
  // reach past the prefix or exceed the bound)
  if (tid == 0) {
    hdr.total = 0;
    hdr.found_seq = -1;
    hdr.found_off = 0;
    hdr.abort_flag = 0;
  }
  __syncthreads();
  {
    long long part = 0;
    for (int i = tid; i < p.num_seqs; i += kAttnThreads) {
      part += suffix_chunks(p, i, pc);
      if (cta == 0) {
        const int raw = p.ctx[i];
        if (raw < 0 || raw > p.ctx_cap || raw <= q.prefix_len) flag_error(p.err, PKVD_ERR_CONTEXT);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL_MASK, part, o);
    if (lane == 0) atomicAdd(reinterpret_cast<unsigned long long*>(&hdr.total), (unsigned long long)part);
  }
  __syncthreads();
  const long long cs = hdr.total;
  const PrefixPlan pl = prefix_plan(q, cs, grid);
  const bool prefix_role = cta < pl.gp;

  // ---- this CTA's work: a prefix range, or a slice of the suffix list
  int sg = 0, sp = 0, c_lo = 0, c_hi = 0;      // prefix role
  long long s0 = 0, s1 = 0;                    // suffix role
  const int cs_cta = cta - pl.gp;
  if (prefix_role) {
    sg = cta / pl.splits;
    sp = cta % pl.splits;
    c_lo = (int)((long long)pc * sp / pl.splits);
    c_hi = (int)((long long)pc * (sp + 1) / pl.splits);
  } else {
    s0 = slice_begin(cs, cs_cta, pl.gs);
    s1 = slice_begin(cs, cs_cta + 1, pl.gs);
    // the row holding the slice's first chunk
    if (s0 < s1) {
      int running = 0;
      for (int base = 0; base < p.num_seqs; base += kAttnThreads) {
        const int i = base + tid;
        const int n = i < p.num_seqs ? suffix_chunks(p, i, pc) : 0;
        int total;
        const int incl = block_incl_scan(n, hdr.scan_warp, total);
        const int excl = running + incl - n;
        if (i < p.num_seqs && n > 0 && excl <= s0 && s0 < excl + n) {
          hdr.found_seq = i;
          hdr.found_off = (int)(s0 - excl);
        }
        running += total;
        __syncthreads();
        if (hdr.found_seq >= 0) break;
      }
    }
  }
  if (tid == 0) pdl_trigger();
  const int nit = prefix_role ? c_hi - c_lo : (int)(s1 - s0);
  if (nit <= 0) return;
  if (!prefix_role && hdr.found_seq < 0) {       // no row holds the slice's first chunk: cannot happen
    if (tid == 0) flag_error(p.err, PKVD_ERR_CONTEXT);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hdr.full[s], 1);
      mbar_init(&hdr.empty[s], p.active_warps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int esz = sizeof(T);

  if (warp == kConsumerWarps) {
    // =============================== producer warp
    const int rows_sg = min(q.sg_rows, p.num_seqs - sg * q.sg_rows);
    int seq = prefix_role ? 0 : hdr.found_seq;             // the row whose table is read
    int ch = prefix_role ? c_lo : hdr.found_off;           // chunk within the part being read
    int nch = prefix_role ? c_hi : suffix_chunks(p, seq, pc);
    int ctx_seq = min(max(p.ctx[seq], 0), p.ctx_cap);
    int seg_first = ch;
    long long row_start = prefix_role ? 0 : s0 - ch;       // suffix: flat index of the row's first chunk
    bool first_seg = true;
    int tb_seq = -1, tb_base = 0, tb_val = -1;
    pdl_wait();
    for (int it = 0; it < nit; ++it) {
      if (!prefix_role) {
        while (ch >= nch && seq + 1 < p.num_seqs) {
          row_start += nch;
          ++seq;
          nch = suffix_chunks(p, seq, pc);
          ctx_seq = min(max(p.ctx[seq], 0), p.ctx_cap);
          ch = 0;
          seg_first = 0;
          first_seg = false;
        }
        if (ch >= nch) break;   // unreachable: the slice never passes the last chunk
      }
      const int stage = it % S;
      const int n = it / S;
      if (n > 0 && !mbar_wait_bounded(&hdr.empty[stage], (n - 1) & 1)) {
        if (lane == 0) { flag_error(p.err, PKVD_ERR_TIMEOUT); hdr.abort_flag = 1; }
        break;
      }
      if (*reinterpret_cast<volatile int*>(&hdr.abort_flag)) break;
      const int token0 = (prefix_role ? ch : pc + ch) * kChunk;
      const int ntok = prefix_role ? kChunk : min(kChunk, ctx_seq - token0);
      const int lb0 = token0 / p.block_size, off0 = token0 % p.block_size;
      if (seq != tb_seq || lb0 < tb_base || lb0 >= tb_base + 32) {
        tb_seq = seq;
        tb_base = lb0;
        const int e = lb0 + lane;
        tb_val = e < p.max_blocks ? p.tables[(int64_t)seq * p.max_blocks + e] : -1;
      }
      const int phys = __shfl_sync(FULL_MASK, tb_val, lb0 - tb_base);
      const bool ok = phys >= 0 && phys < p.num_blocks && ntok > 0;
      const int ncopy = ok ? ntok : 0;
      int flags = 0;
      if (ch == seg_first) flags |= PF_FIRST;
      if (ch == nch - 1 || it == nit - 1) flags |= PF_LAST;
      if (lane == 0) {
        if (!ok && ntok > 0) flag_error(p.err, PKVD_ERR_BLOCK_ID);
        int first_row, rows;
        int64_t rec_first;
        if (prefix_role) {
          first_row = sg * q.sg_rows;
          rows = rows_sg;
          rec_first = ((int64_t)sg * q.max_splits + sp) * q.sg_rows;
        } else {
          first_row = seq;
          rows = 1;
          // the whole suffix of the row in this CTA: its own record;
          // otherwise this CTA's first (slot 0) or last (slot 1) segment
          const bool whole = seg_first == 0 && (row_start + nch - 1) < s1 && row_start >= s0;
          rec_first = whole ? q.rec_rows + seq : q.rec_suffix + (int64_t)cs_cta * 2 + (first_seg ? 0 : 1);
        }
        hdr.meta[stage] = make_int4(first_row, rows, ncopy | (flags << 8), (int)rec_first);
        mbar_arrive_expect_tx(&hdr.full[stage], (uint32_t)(ncopy * 2 * p.row_bytes));
      }
      __syncwarp();
      if (ncopy > 0) {
        uint8_t* sdst = stage_base + stage * stage_bytes;
        // a chunk starts on a 16-token boundary, so it lies in one block
        const int64_t b0 = ((int64_t)phys * p.block_stride + (int64_t)off0 * p.token_stride) * esz;
        if (p.rows_contig) {
          for (int r = lane; r < 2 * ncopy; r += 32) {
            const int kv = r >= ncopy;
            const int t = kv ? r - ncopy : r;
            bulk_g2s(sdst + kv * kChunk * p.rowb + t * p.rowb, (kv ? p.v_base : p.k_base) + b0 +
                     (int64_t)t * p.token_stride * esz, p.row_bytes, &hdr.full[stage]);
          }
        } else {
          const int per = ncopy * p.hkv;
          for (int r = lane; r < 2 * per; r += 32) {
            const int kv = r >= per;
            const int rem = kv ? r - per : r;
            const int t = rem / p.hkv, h = rem % p.hkv;
            bulk_g2s(sdst + kv * kChunk * p.rowb + t * p.rowb + h * D * esz, (kv ? p.v_base : p.k_base) + b0 +
                     ((int64_t)t * p.token_stride + (int64_t)h * p.head_stride) * esz, D * esz, &hdr.full[stage]);
          }
        }
      }
      ++ch;
    }
    // drain: every copy this warp issued has landed before the CTA leaves
    const int last = nit;
    const int first = last > S ? last - S : 0;
    for (int k = first; k < last; ++k) {
      if (!mbar_wait_bounded(&hdr.full[k % S], (k / S) & 1)) {
        if (lane == 0) flag_error(p.err, PKVD_ERR_TIMEOUT);
        break;
      }
    }
    return;
  }

  // ================================== consumer warps
  if (warp >= p.active_warps) return;
  GroupConsumer<T, D> cons;
  for (int it = 0; it < nit; ++it) {
    const int stage = it % S;
    if (!mbar_wait_bounded(&hdr.full[stage], (it / S) & 1)) {
      if (lane == 0) { flag_error(p.err, PKVD_ERR_TIMEOUT); hdr.abort_flag = 1; }
      break;
    }
    const int4 meta = hdr.meta[stage];
    const int ntok = meta.z & 0xff, flags = meta.z >> 8;
    if (flags & PF_FIRST) cons.begin(p, meta.x, meta.y, warp, lane);
    uint8_t* sK = stage_base + stage * stage_bytes;
    uint8_t* sV = sK + kChunk * p.rowb;
    if (ntok > 0) cons.chunk(p, sK, sV, ntok, warp, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&hdr.empty[stage]);
    if (flags & PF_LAST) cons.finish(p, q.rec, meta.w, warp, lane);
  }
}

// ------------------------------------------------------------ merge
// One CTA per row and group of 256 output float4 slices, a programmatic
// dependent of the partition kernel: the row's prefix records (one per
// split of its sub-group) and its suffix records (its own record when one
// suffix CTA held the whole suffix, else one per suffix CTA its suffix
// crosses), combined with the log-sum-exp identity.
template <typename T>
__global__ void __launch_bounds__(256) lse_merge_prefix_kernel(T* __restrict__ out, const PrefixParams q, int D,
                                                               int grid) {
  const PartParams& p = q.p;
  __shared__ int64_t s_rec[kPrefixMaxSplits + kMaxMergeRecords];
  __shared__ int s_n;
  __shared__ long long s_part[2][8];
  const int i = blockIdx.x;
  const int pc = q.prefix_len / kChunk;
  // the suffix geometry from the context lengths (inputs no early-signalling
  // kernel writes), before the dependency wait
  long long before = 0, all = 0;
  for (int r = threadIdx.x; r < p.num_seqs; r += blockDim.x) {
    const int c = suffix_chunks(p, r, pc);
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
  const PrefixPlan pl = prefix_plan(q, C, grid);
  const long long n = suffix_chunks(p, i, pc);
  if (threadIdx.x == 0) {
    int cnt = 0;
    const int sg = i / q.sg_rows, rl = i % q.sg_rows;
    for (int sp = 0; sp < pl.splits; ++sp) s_rec[cnt++] = ((int64_t)sg * q.max_splits + sp) * q.sg_rows + rl;
    if (n > 0) {
      const int G = pl.gs;
      const int a = (int)(((P + 1) * G - 1) / C);
      const int b = (int)(((P + n) * G - 1) / C);
      const bool a_at_start = (C * a) / G == P;
      if (a == b) {
        s_rec[cnt++] = q.rec_rows + i;                      // one suffix CTA held the whole suffix
      } else {
        for (int c = a; c <= b && cnt < kPrefixMaxSplits + kMaxMergeRecords; ++c) {
          if (C < G && (C * c) / G >= (C * (c + 1)) / G) continue;
          s_rec[cnt++] = q.rec_suffix + (int64_t)c * 2 + ((c == a && !a_at_start) ? 1 : 0);
        }
      }
    }
    s_n = cnt;
  }
  __syncthreads();
  const int nrec = s_n;
  pdl_wait();                       // the partition kernel's records
  pdl_trigger();
  T* orow = out + (int64_t)i * p.hq * D;
  // four adjacent lanes share one float4 output slice, each taking every
  // fourth record; their states are combined with shuffles
  constexpr int kParts = 4;
  const int Q = D / 4;
  constexpr int R = 8;
  const int nslots = p.hq * Q * kParts;
  for (int base = blockIdx.y * blockDim.x; base < nslots; base += gridDim.y * blockDim.x) {
    const int t = base + threadIdx.x;                 // whole warps iterate together
    const int sl = t / kParts, part = t % kParts;
    const bool live = t < nslots;
    const int h = live ? sl / Q : 0, d4 = live ? (sl % Q) * 4 : 0;
    float M = -INFINITY, L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = part; live && k0 < nrec; k0 += R * kParts) {
      float mk[R], lk[R];
      float4 ak[R];
#pragma unroll
      for (int e = 0; e < R; ++e) {
        const int k = k0 + e * kParts;
        mk[e] = -INFINITY;
        lk[e] = 0.f;
        ak[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < nrec) {
          const float* r = q.rec + (s_rec[k] * p.hq + h) * (D + 4);
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
#pragma unroll
    for (int off = 1; off < kParts; off <<= 1) {
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
      const float inv = L > 0.f ? 1.f / L : 0.f;
      T* dst = orow + h * D + d4;
      dst[0] = DT<T>::from_f(o.x * inv);
      dst[1] = DT<T>::from_f(o.y * inv);
      dst[2] = DT<T>::from_f(o.z * inv);
      dst[3] = DT<T>::from_f(o.w * inv);
    }
  }
}

int sg_rows_of(int group) { return group >= kPrefixQueries ? 1 : kPrefixQueries / group; }

int max_splits_of(int prefix_len) {
  const int pc = prefix_len / kChunk;
  return pc < kPrefixMaxSplits ? pc : kPrefixMaxSplits;
}

template <typename T, int D>
cudaError_t launch_prefix_t(const AttnArgs& a, const PrefixParams& q, cudaStream_t stream) {
  const size_t smem = smem_header_bytes() + (size_t)q.p.stages * 2 * kChunk * q.p.rowb;
  auto kern = paged_decode_prefix_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(a.grid), dim3(kAttnThreads), smem, stream, q);
  if (e != cudaSuccess) return e;
  const int groups = (a.num_q_heads * (D / 4) * 4 + 255) / 256;     // four lanes per output slice
  return launch_pdl(lse_merge_prefix_kernel<T>, dim3((unsigned)a.num_seqs, (unsigned)groups), dim3(256), 0, stream,
                    static_cast<T*>(a.out), q, D, a.grid);
}

}  // namespace

bool prefix_path_usable(int dtype, int head_dim, int num_kv_heads, int num_q_heads, int num_seqs, int grid,
                        int prefix_len, int window) {
  if (dtype == PKVD_F32 || num_kv_heads != 8 || (head_dim != 64 && head_dim != 128)) return false;
  if (num_q_heads % num_kv_heads) return false;
  const int group = num_q_heads / num_kv_heads;
  if (group < 1 || group > 8 || window > 0 || prefix_len < kChunk || num_seqs < 2) return false;
  const int sg = sg_rows_of(group);
  const int nsg = (num_seqs + sg - 1) / sg;
  return nsg < grid;                               // leaves at least one CTA for the suffixes
}

size_t prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int grid,
                              int prefix_len) {
  const int group = num_kv_heads > 0 ? num_q_heads / num_kv_heads : 1;
  const int sg = sg_rows_of(group < 1 ? 1 : group);
  const long long nsg = (num_seqs + sg - 1) / sg;
  const long long recs = nsg * max_splits_of(prefix_len) * sg + 2LL * grid + num_seqs;
  return (size_t)recs * num_q_heads * (head_dim + 4) * sizeof(float);
}

cudaError_t launch_attention_prefix(const AttnArgs& a, int prefix_len, cudaStream_t stream) {
  PrefixParams q;
  q.p = part_params(a, nullptr);
  q.prefix_len = prefix_len;
  q.sg_rows = sg_rows_of(q.p.G);
  q.nsg = (a.num_seqs + q.sg_rows - 1) / q.sg_rows;
  q.max_splits = max_splits_of(prefix_len);
  q.rec = static_cast<float*>(a.workspace);
  q.rec_suffix = (int64_t)q.nsg * q.max_splits * q.sg_rows;
  q.rec_rows = q.rec_suffix + 2LL * a.grid;
  if (a.dtype == PKVD_F16)
    return a.head_dim == 64 ? launch_prefix_t<__half, 64>(a, q, stream) : launch_prefix_t<__half, 128>(a, q, stream);
  return a.head_dim == 64 ? launch_prefix_t<__nv_bfloat16, 64>(a, q, stream)
                          : launch_prefix_t<__nv_bfloat16, 128>(a, q, stream);
}

}  // namespace pkvd
