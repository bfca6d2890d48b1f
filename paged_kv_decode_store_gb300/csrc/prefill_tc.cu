// Varlen paged prefill attention on the 5th-generation tensor cores
// (tcgen05: operands in shared memory, accumulators in tensor memory).
//
// Same operation as prefill.cu (nano-vllm "Model Runner" notes, sections
// "prefix cache" and "prefill and decode": cu_seqlens_q / cu_seqlens_k
// describe the batch, new token j of sequence i sits at position
// (k_len_i - q_len_i) + j and attends causally to positions 0..p of its
// sequence through the block table).
//
// One CTA per (KV head, sequence, pair of 128-row Q tiles); row = token * G +
// query head of the group, so every K/V tile serves the whole GQA group, and
// both Q tiles of the pair share each K/V tile the CTA loads.  Pairs are
// counted from the end of each sequence.  While the batch's K/V fits in L2
// the heaviest pairs of every sequence start first; otherwise CTAs of one
// (sequence, KV head) run together so that its K/V tiles stay in L2.  Twelve warps with fixed roles:
//   warps 0-3, 4-7  softmax of Q tile 0 and 1: thread r owns query row r =
//              TMEM lane r.  Loads its Q row into shared memory, then per
//              128-key tile reads its row of S from TMEM, masks (causal,
//              window), keeps a running max (re-based only when it grows by
//              more than 2^8, so O is rarely rescaled), writes P = 2^(S - max)
//              as packed 16-bit pairs into TMEM, and at the end reads O from
//              TMEM, divides by the row sum and stores it.
//   warps 8, 10  producers of K and of V: TMA (cp.async.bulk.tensor, 128-byte
//              swizzle) of each tile's rows, one box per (cache block
//              segment, 64-column half); the V warp zeroes rows outside the
//              pair's key range in the first and last tiles before releasing
//              them.
//   warps 9, 11  MMA for Q tile 0 and 1 (warp 9 also allocates the 512 TMEM
//              columns): one thread each issues S = Q K^T (M 128, N 128 keys,
//              K = head_dim) and O += P V (M 128, N = head_dim, K 128 keys, P
//              from TMEM) for its Q tile with tcgen05.mma kind::f16 (fp32
//              accumulate), and signals mbarriers with tcgen05.commit.
// Keys outside a row's range are masked in S; segments whose block id is bad
// read as zeros.
//
// Shared-memory operand layout (K-major, 128-byte swizzle): a 128-row tile of
// 64 16-bit columns is 128 rows of 128 bytes, 16-byte chunk c of row r at
// r*128 + ((c ^ (r % 8)) * 16); head_dim 128 uses two such halves.  Q and K
// are read K-major (stride between 8-row groups 1024 B); V is read
// MN-major (head_dim contiguous: 1024 B between 8-key groups, one half-tile
// between 64-column halves).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace pkvd {

namespace {

constexpr int kTcRows = 128;          // M: query rows per Q tile (two Q tiles per CTA)
constexpr int kTcKeys = 128;          // keys per K/V tile
constexpr int kTcThreads = 384;       // 2 x 4 softmax warps, K producer, MMA 0, V producer, MMA 1
constexpr int kGroup = 128;           // softmax threads per Q tile (one per row)
constexpr int kProducerWarp = 8, kMmaWarp = 9, kVProducerWarp = 10, kMmaWarp1 = 11;
constexpr uint32_t kHalf = 128u * 128u;   // one 128-row x 64-column 16-bit half tile
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S of Q tile g at [128 g, 128 g + 128) (P of that tile is written
// over its first 64 columns once S is read); O of Q tile g at [256 + g D, 256 + g D + D)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr float kRebase = 8.f;        // re-base the running max when it grows by > 2^8

template <int D>
struct TcLayout {
  // K and V stages: as many as shared memory holds (K three and V two tiles
  // ahead of the tensor cores for head_dim 128, four each for 64)
  static constexpr int kKStages = D == 64 ? 4 : 3, kVStages = D == 64 ? 4 : 2;
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kQ = 0;                                    // 2 Q tiles
  static constexpr uint32_t kK = kQ + 2 * kHalves * kHalf;             // kKStages stages
  static constexpr uint32_t kV = kK + kKStages * kHalves * kHalf;      // kVStages stages
  static constexpr uint32_t kBar = kV + kVStages * kHalves * kHalf;
  // + alignment slack; at least 120 KB so that one CTA (which holds all 512
  // TMEM columns) is resident per SM
  static constexpr uint32_t kBytes = kBar + 512 + 1024 > 122880u ? kBar + 512 + 1024 : 122880u;
};

// mbarrier slots (8 bytes each) after kBar.  Per-Q-tile barriers take + g.
// Every barrier's next phase depends on its waiter having passed the current
// one, so no waiter ever sees a barrier two phases ahead.
enum : int {
  kKFull = 0, kKEmpty = 4, kVFull = 8, kVReady = 12, kVEmpty = 16, kQFull = 20, kSFull = 22, kPFull = 24,
  kPVDone = 26, kSRead = 28, kDrain = 30, kNumBars = 32
};
// With head_dim 64 TMEM also holds a separate P buffer per Q tile at
// [384 + 64 g, 448 + 64 g): the next S may then be computed as soon as the
// softmax has read the current one (S-read barrier) instead of after its PV.
constexpr uint32_t kColP64 = 384;
constexpr uint32_t kTmemSlot = 8 * kNumBars;   // the allocated TMEM base address

struct TcParams {
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  void* out;
  const void* q;
  const int32_t* tables;
  int max_blocks;
  int64_t num_blocks;
  int block_size;
  int seg_rows;          // rows per TMA box: min(block_size, 128)
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q;
  int hq;
  int group;
  int tile_tokens;
  int pairs;             // Q-tile pairs per (sequence, KV head): the grid is pairs x Hkv x num_seqs
  int num_seqs;
  int64_t l2_bytes;      // the device's L2 size, for the CTA order
  float scale_log2;
  int window;
  int32_t* err;
};

// Spin (test_wait) until the phase with this parity has completed; false
// after 2 s without it (the caller flags PKVD_ERR_TIMEOUT).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity);
__device__ __forceinline__ bool mbar_poll_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t spin = 0;; ++spin) {
    if (mbar_test(bar, parity)) return true;
    if ((spin & 255u) == 255u && globaltimer_ns() - t0 > 2000000000ull) return false;
  }
}

// Non-blocking: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ int tc_window_start(int c, int window) {
  return (window > 0 && c > window) ? c - window : 0;
}

__device__ __forceinline__ float tc_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (one instruction on sm_100-family parts).
__device__ __forceinline__ float tc_max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pair arithmetic on two fp32 lanes (one instruction each).
__device__ __forceinline__ void tc_fma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  unsigned long long a, bb, cc, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(bb) : "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(bb), "l"(cc));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}
__device__ __forceinline__ void tc_add2(float& d0, float& d1, float a0, float a1) {
  unsigned long long a, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(d0), "f"(d1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(d), "l"(a));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}

// ------------------------------------------------------------ tcgen05 PTX
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16, one CTA.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16: A (M x 16) lane i = row i,
// 16-bit pairs along K packed in 32-bit columns.
__device__ __forceinline__ void tc_mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: 128-byte swizzle, version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (0 f16, 1 bf16), A K-major, B K-major (b_mn = 0) or MN-major.
__host__ __device__ constexpr uint32_t tc_idesc(uint32_t fmt, uint32_t n, uint32_t b_mn) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (b_mn << 16) | ((n >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);
}

// 4-D tiled TMA load: coordinates (column, kv head, row in block, block).
__device__ __forceinline__ void tma_load4(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled half tile.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <typename T, int D>
// 12 warps: an SM sub-partition holds three of them, so at most 168 registers a thread
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
  using L = TcLayout<D>;
  constexpr int H = L::kHalves;
  constexpr int kKStages = L::kKStages, kVStages = L::kVStages;
  constexpr bool kSepP = D == 64;                        // P in its own TMEM columns
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;          // 1024-byte aligned: whole swizzle atoms
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + L::kBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();      // the cache rows of this step come from the store kernel
  pdl_trigger();

  // CTA order: while the batch's K/V fits in L2, KV head fastest and pair
  // slowest (the heaviest causal work of every sequence first); otherwise
  // pair fastest, so CTAs resident together share one (sequence, KV head) and
  // its K/V tiles stay in L2.  Every CTA takes the same decision; the
  // sequence lengths of both candidate orders are loaded together with the
  // batch's key count (one round trip).
  // the grid is (KV heads, sequences, pairs); lin is the linear CTA index
  const int nh = (int)gridDim.x;
  const int lin = blockIdx.x + nh * (blockIdx.y + p.num_seqs * blockIdx.z);
  const int seq_a = (lin / nh) % p.num_seqs, seq_b = lin / (p.pairs * nh);
  const int total_keys = p.cu_k[p.num_seqs];
  const int qa0 = p.cu_q[seq_a], qa1 = p.cu_q[seq_a + 1], ka0 = p.cu_k[seq_a], ka1 = p.cu_k[seq_a + 1];
  const int qb0 = p.cu_q[seq_b], qb1 = p.cu_q[seq_b + 1], kb0 = p.cu_k[seq_b], kb1 = p.cu_k[seq_b + 1];
  const bool by_cost = (int64_t)total_keys * nh * D * 4 <= p.l2_bytes;   // K and V, 16-bit
  const int seq = by_cost ? seq_a : seq_b;
  const int hk = by_cost ? lin % nh : (lin / p.pairs) % nh;
  const int zpair = by_cost ? lin / (nh * p.num_seqs) : lin % p.pairs;
  const int q0 = by_cost ? qa0 : qb0, q1 = by_cost ? qa1 : qb1;
  const int klen = by_cost ? ka1 - ka0 : kb1 - kb0;
  const int qlen = q1 - q0;
  if (q0 < 0 || qlen < 0 || klen < qlen || q1 > p.total_q ||
      (int64_t)klen > (int64_t)p.max_blocks * p.block_size) {
    if (threadIdx.x == 0 && zpair == 0 && hk == 0) flag_error(p.err, PKVD_ERR_CONTEXT);
    return;
  }
  if (zpair == 0 && hk == 0 && threadIdx.x == 0 && qlen > 2 * p.pairs * p.tile_tokens)
    flag_error(p.err, PKVD_ERR_CONTEXT);   // longer than max_seqlen_q: the earliest tokens are not computed
  // Q tile g = 1 holds the later tokens (tile 2 zpair counted from the end),
  // g = 0 the tile before it (may be empty).
  const int Tt = p.tile_tokens, G = p.group, cached = klen - qlen;
  int tb[2], te[2], lo_g[2], hi_g[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    te[g] = qlen - (2 * zpair + 1 - g) * Tt;
    tb[g] = max(0, te[g] - Tt);
    lo_g[g] = tc_window_start(cached + tb[g] + 1, p.window);   // first key the tile's rows read
    hi_g[g] = cached + te[g] - 1;                               // last key
  }
  if (te[1] <= 0) return;
  const bool has0 = te[0] > 0;
  const int lo = has0 ? lo_g[0] : lo_g[1], hi = hi_g[1];        // union of both tiles' keys
  const int kt_first = lo / kTcKeys;
  const int n = hi / kTcKeys - kt_first + 1;                    // K/V tiles of the CTA
  int gf[2], gn[2];                                             // each Q tile's K/V tiles
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    gf[g] = lo_g[g] / kTcKeys - kt_first;
    gn[g] = (g == 0 && !has0) ? 0 : hi_g[g] / kTcKeys - lo_g[g] / kTcKeys + 1;
  }
  const int32_t* table = p.tables + (int64_t)seq * p.max_blocks;
  const int nseg = kTcKeys / p.seg_rows;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(&bars[i], (i == kQFull || i == kQFull + 1 || i == kPFull || i == kPFull + 1 || i == kSRead ||
                           i == kSRead + 1) ? (uint32_t)kGroup
                          : kSepP && ((i >= kKEmpty && i < kKEmpty + 4) || (i >= kVEmpty && i < kVEmpty + 4)) ? 2u
                                                                                                              : 1u);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(base + L::kBar + kTmemSlot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + L::kBar + kTmemSlot);

  if (warp == kProducerWarp || warp == kVProducerWarp) {
    // ------------------------------------------------------------ producers
    // Warp 8 copies the K tiles, warp 10 the V tiles, each as fast as its
    // ring of stages frees up (one warp issuing both was the bottleneck: a
    // tile of 16-row segments takes 16 TMA issues per operand).  Lane 0 polls
    // for the next free stage; lane s looks up (three tiles ahead) and copies
    // segment s of the tile.  A V tile with rows outside [lo, hi] (the first
    // and last tiles) is waited for here and those rows zeroed before the tile
    // is released (V ready), so rows outside every query's range never weigh in.
    const bool is_v = warp == kVProducerWarp;
    const int stages = is_v ? kVStages : kKStages;
    const int full0 = is_v ? kVFull : kKFull, empty0 = is_v ? kVEmpty : kKEmpty;
    const uint32_t ring = base + (is_v ? L::kV : L::kK);
    const CUtensorMap* map = is_v ? &p.tmap_v : &p.tmap_k;
    const uint32_t box = (uint32_t)p.seg_rows * 128u;
    int t = 0;
    bool ok = true;
    if (lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
    uint64_t t_start = globaltimer_ns();       // the last progress
    constexpr int kNone = INT_MIN;             // a segment that misses [lo, hi]: nothing to load
    auto fetch = [&](int tt) -> int {
      if (tt >= n || lane >= nseg) return kNone;
      const int ks = (kt_first + tt) * kTcKeys + lane * p.seg_rows;
      if (ks > hi || ks + p.seg_rows - 1 < lo) return kNone;
      return __ldg(table + ks / p.block_size);
    };
    // each lane's block id of tiles t .. t + 3
    int b0 = fetch(0), b1 = fetch(1), b2 = fetch(2), b3 = fetch(3);
    while (t < n) {
      int go = 0;   // 1: issue tile t, -1: gave up
      if (lane == 0) {
        if (t < stages || mbar_test(&bars[empty0 + t % stages], ((t / stages) - 1) & 1)) go = 1;
        else if (globaltimer_ns() - t_start > 2000000000ull) go = -1;
      }
      go = __shfl_sync(FULL_MASK, go, 0);
      if (go < 0) {
        ok = false;
        break;
      }
      if (go == 0) continue;
      const bool good = b0 != kNone && b0 >= 0 && b0 < p.num_blocks;
      const uint32_t loaded = __ballot_sync(FULL_MASK, good);
      if (!is_v && __ballot_sync(FULL_MASK, b0 != kNone && !good) && lane == 0) flag_error(p.err, PKVD_ERR_BLOCK_ID);
      const int stg = t % stages;
      uint64_t* bar = &bars[full0 + stg];
      const uint32_t dst0 = ring + stg * H * kHalf;
      const int kbase = (kt_first + t) * kTcKeys;
      // a segment with a bad block id reads as zeros (like the mma.sync path)
      if (b0 != kNone && !good) {
        for (int h = 0; h < H; ++h)
          for (uint32_t o = 0; o < box; o += 16) st_shared_v4(dst0 + h * kHalf + lane * box + o, make_uint4(0u, 0u, 0u, 0u));
        fence_proxy_async_smem();
      }
      __syncwarp();
      // lane 0 announces the bytes, then lane s copies segment s (in parallel)
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(loaded) * box * H);
      __syncwarp();
      if ((loaded >> lane) & 1u) {
        const int ks = kbase + lane * p.seg_rows;
#pragma unroll
        for (int h = 0; h < H; ++h) tma_load4(dst0 + h * kHalf + lane * box, map, h * 64, hk, ks % p.block_size, b0, bar);
      }
      if (is_v) {
        // V ready: at once, or, for an edge tile, once its rows outside [lo, hi] are zero
        if (kbase < lo || kbase + kTcKeys - 1 > hi) {
          if (lane == 0) ok = mbar_wait_bounded(bar, (t / stages) & 1);
          if (!(ok = __shfl_sync(FULL_MASK, ok, 0))) {
            ++t;
            break;
          }
          for (int rr = lane; rr < kTcKeys; rr += 32) {
            const int kp = kbase + rr;
            if (kp >= lo && kp <= hi) continue;
            for (int h = 0; h < H; ++h)
              for (int c = 0; c < 8; ++c) st_shared_v4(dst0 + h * kHalf + rr * 128 + c * 16, make_uint4(0u, 0u, 0u, 0u));
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) mbar_arrive(&bars[kVReady + stg]);
      }
      ++t;
      b0 = b1;
      b1 = b2;
      b2 = b3;
      b3 = fetch(t + 3);
      if (lane == 0) t_start = globaltimer_ns();
    }
    if (!ok && lane == 0) {
      // gave up: let this warp's copies still in flight land before the CTA leaves
      flag_error(p.err, PKVD_ERR_TIMEOUT);
      for (int u = max(0, t - stages); u < t; ++u) mbar_wait_bounded(&bars[full0 + u % stages], (u / stages) & 1);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp1) {
    // ---------------------------------------------------------------- MMA
    // head_dim 64: one issuing thread per Q tile (warp 9: tile 0, warp 11:
    // tile 1), so a thread that stalls while the tensor pipe takes one tile's
    // products never holds up the other's.  Tile g's sequence: S_g(j) once
    // K(j) has landed (and Q_g, for j = 0) and the softmax has read
    // S_g(j - 1) (P_g has its own columns), so S_g(j) is issued before
    // PV_g(j - 1); PV_g(j) once P_g(j) and V(j) are ready.  A K or V stage is
    // released when both Q tiles are done with it: its empty barrier counts
    // two arrivals, and a tile that only one Q tile uses gets both from that
    // tile's commits.
    if constexpr (kSepP) {
      const int g = warp == kMmaWarp ? 0 : 1, o = 1 - g;
      if (lane == 0 && gn[g] > 0) {
        constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
        constexpr uint32_t id_s = tc_idesc(fmt, kTcKeys, 0), id_pv = tc_idesc(fmt, D, 1);
        bool ok = true;
        auto wait = [&](int bar, uint32_t parity) {
          if (ok) ok = mbar_poll_bounded(&bars[bar], parity);
        };
        auto release = [&](int empty, int t) {
          tc_commit(&bars[empty]);
          if (!(t >= gf[o] && t < gf[o] + gn[o])) tc_commit(&bars[empty]);   // the other tile's share
        };
        auto issue_s = [&](int j) {
          const int t = gf[g] + j;
          wait(kKFull + t % kKStages, (t / kKStages) & 1);
          if (!ok) return;
          tc_fence_after();
          const uint32_t qb = base + L::kQ + g * H * kHalf;
          const uint32_t kb = base + L::kK + (t % kKStages) * H * kHalf;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
            tc_mma(tmem + kColS + g * kTcKeys, smem_desc(qb + off, 16, 1024), smem_desc(kb + off, 16, 1024), id_s, k > 0);
          }
          tc_commit(&bars[kSFull + g]);
          release(kKEmpty + t % kKStages, t);
        };
        auto issue_pv = [&](int j) {
          const int t = gf[g] + j;
          wait(kPFull + g, j & 1);
          wait(kVFull + t % kVStages, (t / kVStages) & 1);
          wait(kVReady + t % kVStages, (t / kVStages) & 1);
          if (!ok) return;
          tc_fence_after();
          const uint32_t vb = base + L::kV + (t % kVStages) * H * kHalf;
#pragma unroll
          for (int k = 0; k < kTcKeys / 16; ++k)      // 16 keys = 8 packed P columns per step
            tc_mma_tmem_a(tmem + kColO + g * D, tmem + kColP64 + g * 64 + k * 8, smem_desc(vb + k * 2048, kHalf, 1024),
                          id_pv, (j > 0 || k > 0) ? 1u : 0u);
          tc_commit(&bars[kPVDone + g]);
          release(kVEmpty + t % kVStages, t);
        };
        wait(kQFull + g, 0);
        issue_s(0);
        for (int j = 0; j < gn[g] && ok; ++j) {
          if (j + 1 < gn[g]) {
            wait(kSRead + g, j & 1);
            issue_s(j + 1);
          }
          issue_pv(j);
        }
        if (!ok) {
          flag_error(p.err, PKVD_ERR_TIMEOUT);
          tc_commit(&bars[kDrain + g]);      // wait for the tensor-core work already issued
          mbar_wait_bounded(&bars[kDrain + g], 0);
        }
      }
    } else if (warp == kMmaWarp) {
      // head_dim 128: one thread issues whatever is ready for either Q tile
      // (S_g(j) needs PV_g(j - 1) finished, so a second issuer only
      // interleaves the two tiles' products and delays both)
      if (lane == 0) {
        constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
        constexpr uint32_t id_s = tc_idesc(fmt, kTcKeys, 0), id_pv = tc_idesc(fmt, D, 1);
        int js[2] = {0, 0}, jp[2] = {0, 0};
        bool ok = true;
        uint64_t t_start = globaltimer_ns();        // the last progress
        auto uses = [&](int g, int t) { return t >= gf[g] && t < gf[g] + gn[g]; };
        while (ok && (jp[0] < gn[0] || jp[1] < gn[1])) {
          bool progressed = false;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (js[g] < gn[g]) {
              const int t = gf[g] + js[g];
              const bool ready = (js[g] == 0 ? mbar_test(&bars[kQFull + g], 0)
                                             : mbar_test(&bars[kPVDone + g], (js[g] - 1) & 1)) &&
                                 mbar_test(&bars[kKFull + t % kKStages], (t / kKStages) & 1);
              if (ready) {
                tc_fence_after();
                const uint32_t qb = base + L::kQ + g * H * kHalf;
                const uint32_t kb = base + L::kK + (t % kKStages) * H * kHalf;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                  const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
                  tc_mma(tmem + kColS + g * kTcKeys, smem_desc(qb + off, 16, 1024), smem_desc(kb + off, 16, 1024),
                         id_s, k > 0);
                }
                tc_commit(&bars[kSFull + g]);
                const int o = 1 - g;
                if (!uses(o, t) || js[o] > t - gf[o]) tc_commit(&bars[kKEmpty + t % kKStages]);
                ++js[g];
                progressed = true;
              }
            }
            if (jp[g] < js[g]) {
              const int t = gf[g] + jp[g];
              const bool ready = mbar_test(&bars[kPFull + g], jp[g] & 1) &&
                                 mbar_test(&bars[kVFull + t % kVStages], (t / kVStages) & 1) &&
                                 mbar_test(&bars[kVReady + t % kVStages], (t / kVStages) & 1);
              if (ready) {
                tc_fence_after();
                const uint32_t vb = base + L::kV + (t % kVStages) * H * kHalf;
#pragma unroll
                for (int k = 0; k < kTcKeys / 16; ++k)      // 16 keys = 8 packed P columns per step
                  tc_mma_tmem_a(tmem + kColO + g * D, tmem + kColS + g * kTcKeys + k * 8,
                                smem_desc(vb + k * 2048, kHalf, 1024), id_pv, (jp[g] > 0 || k > 0) ? 1u : 0u);
                tc_commit(&bars[kPVDone + g]);
                const int o = 1 - g;
                if (!uses(o, t) || jp[o] > t - gf[o]) tc_commit(&bars[kVEmpty + t % kVStages]);
                ++jp[g];
                progressed = true;
              }
            }
          }
          if (progressed) t_start = globaltimer_ns();
          else if (globaltimer_ns() - t_start > 2000000000ull) ok = false;
        }
        if (!ok) {
          flag_error(p.err, PKVD_ERR_TIMEOUT);
          tc_commit(&bars[kDrain]);          // wait for the tensor-core work already issued
          mbar_wait_bounded(&bars[kDrain], 0);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Group g (warps 4g .. 4g + 3) owns Q tile g; thread r owns its row r =
    // TMEM lane r: it reads the row's S from TMEM, masks (causal, window),
    // keeps a running max re-based only when it grows by more than 2^8
    // (exact; O is rescaled in TMEM rarely), writes P = 2^(s - max) as packed
    // 16-bit pairs over the first 64 S columns, and at the end reads O,
    // divides by the row sum and stores it.
    const int g = warp >> 2, r = threadIdx.x & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // this group's tile, as scalars (no runtime-indexed arrays)
    const int my_tb = g ? tb[1] : tb[0], my_te = g ? te[1] : te[0];
    const int my_gf = g ? gf[1] : gf[0], my_gn = g ? gn[1] : gn[0];
    if (my_gn > 0) {
      const int qrows = (my_te - my_tb) * G;
      const bool live = r < qrows;
      const int tt = live ? r / G : 0, gi = live ? r - (r / G) * G : 0;
      const int pr = cached + my_tb + tt;          // padding rows mirror row 0
      const int wr = tc_window_start(pr + 1, p.window);
      {
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const T*>(p.q) + ((int64_t)(q0 + my_tb + tt) * p.hq + (int64_t)hk * G + gi) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
          st_shared_v4(base + L::kQ + (g * H + (c >> 3)) * kHalf + swz(r, c & 7), v);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[kQFull + g]);
      }
      const uint32_t s_addr = tmem + lane_base + kColS + g * kTcKeys;
      const uint32_t o_addr = tmem + lane_base + kColO + g * D;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < my_gn; ++j) {
        const int kbase = (kt_first + my_gf + j) * kTcKeys;
        const int c_lo = max(wr - kbase, 0), c_hi = min(pr - kbase, kTcKeys - 1);
        const bool row_full = c_lo == 0 && c_hi == kTcKeys - 1;
        uint32_t mw[kTcKeys / 32];
#pragma unroll
        for (int w = 0; w < kTcKeys / 32; ++w) {
          const int a = min(max(c_lo - 32 * w, 0), 32), z = min(max(c_hi + 1 - 32 * w, 0), 32);
          mw[w] = (z == 32 ? 0xffffffffu : ((1u << z) - 1u)) & ~(a == 32 ? 0xffffffffu : ((1u << a) - 1u));
        }
        ok = __all_sync(FULL_MASK, mbar_wait_bounded(&bars[kSFull + g], j & 1));
        if (!ok) break;
        tc_fence_after();
        float v[kTcKeys];
#pragma unroll
        for (int c4 = 0; c4 < kTcKeys / 32; ++c4) tmem_ld32(s_addr + c4 * 32, v + c4 * 32);
        tmem_ld_wait();
        if constexpr (kSepP) {
          tc_fence_before();
          mbar_arrive(&bars[kSRead + g]);            // the next S may overwrite these columns
        }
        // raw scores: the scale (> 0) is applied inside the exponent, so the
        // row max is taken over the raw values and scaled once
        if (!row_full) {
#pragma unroll
          for (int c = 0; c < kTcKeys; ++c)
            v[c] = ((mw[c >> 5] >> (c & 31)) & 1u) ? v[c] : -INFINITY;
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTcKeys; c += 8) {
          mx0 = tc_max3(mx0, v[c], v[c + 1]);
          mx1 = tc_max3(mx1, v[c + 2], v[c + 3]);
          mx2 = tc_max3(mx2, v[c + 4], v[c + 5]);
          mx3 = tc_max3(mx3, v[c + 6], v[c + 7]);
        }
        const float mt = fmaxf(tc_max3(mx0, mx1, mx2), mx3) * p.scale_log2;
        const bool rebase = mt > m_ref + kRebase;
        const bool scale_o = rebase && m_ref != -INFINITY;
        const float alpha = scale_o ? tc_ex2(m_ref - mt) : 1.f;
        if (rebase) m_ref = mt;
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        uint32_t pk[kTcKeys / 2];
        float rs0 = 0.f, rs1 = 0.f, rs2 = 0.f, rs3 = 0.f;
#pragma unroll
        for (int c = 0; c < kTcKeys; c += 4) {
          // 2^(scale * s - mu) for two keys per packed FMA; masked keys give 2^-inf = 0
          float a0, a1, a2, a3;
          tc_fma2(a0, a1, v[c], v[c + 1], p.scale_log2, -mu);
          tc_fma2(a2, a3, v[c + 2], v[c + 3], p.scale_log2, -mu);
          const float e0 = tc_ex2(a0), e1 = tc_ex2(a1), e2 = tc_ex2(a2), e3 = tc_ex2(a3);
          if (c & 4) tc_add2(rs2, rs3, e0, e1), tc_add2(rs2, rs3, e2, e3);
          else tc_add2(rs0, rs1, e0, e1), tc_add2(rs0, rs1, e2, e3);
          pk[c / 2] = Mma<T>::pack(e0, e1);
          pk[c / 2 + 1] = Mma<T>::pack(e2, e3);
        }
        l = l * alpha + ((rs0 + rs1) + (rs2 + rs3));
        if constexpr (kSepP) {
          // the P buffer and O are free once PV(j - 1) has finished
          if (j > 0) {
            ok = __all_sync(FULL_MASK, mbar_wait_bounded(&bars[kPVDone + g], (j - 1) & 1));
            if (!ok) break;
            tc_fence_after();
          }
        }
        // PV(j - 1) has finished: O may be rescaled
        if (__any_sync(FULL_MASK, scale_o)) {
#pragma unroll 1
          for (int c4 = 0; c4 < D / 32; ++c4) {
            float o[32];
            tmem_ld32(o_addr + c4 * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(o_addr + c4 * 32, o);
          }
        }
        const uint32_t p_addr = kSepP ? tmem + lane_base + kColP64 + g * 64 : s_addr;
        tmem_st32(p_addr, reinterpret_cast<const float*>(pk));
        tmem_st32(p_addr + 32, reinterpret_cast<const float*>(pk + 32));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[kPFull + g]);
      }
      if (ok) ok = __all_sync(FULL_MASK, mbar_wait_bounded(&bars[kPVDone + g], (my_gn - 1) & 1));
      if (ok) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T* dst = static_cast<T*>(p.out) + ((int64_t)(q0 + my_tb + tt) * p.hq + (int64_t)hk * G + gi) * D;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          float o[32];
          tmem_ld32(o_addr + c4 * 32, o);
          tmem_ld_wait();
          if (live) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint4 w;
              w.x = Mma<T>::pack(o[c8 * 8 + 0] * inv, o[c8 * 8 + 1] * inv);
              w.y = Mma<T>::pack(o[c8 * 8 + 2] * inv, o[c8 * 8 + 3] * inv);
              w.z = Mma<T>::pack(o[c8 * 8 + 4] * inv, o[c8 * 8 + 5] * inv);
              w.w = Mma<T>::pack(o[c8 * 8 + 6] * inv, o[c8 * 8 + 7] * inv);
              *reinterpret_cast<uint4*>(dst + c4 * 32 + c8 * 8) = w;
            }
          }
        }
      } else if (lane == 0) {
        flag_error(p.err, PKVD_ERR_TIMEOUT);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

// The driver's tensor-map encoder (one entry point for every device and
// context).  Threads racing on the first lookup all store the same pointer.
std::atomic<EncodeTiled> g_encode_fn{nullptr};

EncodeTiled encode_fn() {
  EncodeTiled fn = g_encode_fn.load(std::memory_order_acquire);
  if (fn) return fn;
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess) {
    fn = reinterpret_cast<EncodeTiled>(f);
    g_encode_fn.store(fn, std::memory_order_release);
  }
  return fn;
}

// Tensor map over one cache ([num_blocks, block_size, Hkv, D] with element
// strides), box = 64 columns x 1 head x seg_rows rows x 1 block, 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* base, const pkvd_cache& c, int seg_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)c.head_dim, (cuuint64_t)c.num_kv_heads, (cuuint64_t)c.block_size,
                              (cuuint64_t)c.num_blocks};
  const cuuint64_t strides[3] = {(cuuint64_t)c.head_stride * 2, (cuuint64_t)c.token_stride * 2,
                                 (cuuint64_t)c.block_stride * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)seg_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt = c.dtype == PKVD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <typename T, int D>
cudaError_t launch_tc_typed(const TcParams& prm, dim3 grid, cudaStream_t stream) {
  constexpr int smem = TcLayout<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(prefill_tc_kernel<T, D>, grid, dim3(kTcThreads), smem, stream, prm);
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& a) {
  const pkvd_cache& c = a.cache;
  if (c.dtype != PKVD_F16 && c.dtype != PKVD_BF16) return false;
  if (c.head_dim != 64 && c.head_dim != 128) return false;
  if (c.block_size < 8) return false;
                       // a TMA box must fill whole 8-row swizzle atoms
  const int G = a.num_q_heads / c.num_kv_heads;
  if (G < 1 || G > kTcRows) return false;
  if ((reinterpret_cast<uintptr_t>(a.out) & 15u) || (reinterpret_cast<uintptr_t>(a.q) & 15u)) return false;
  // the box walks the cache as nested dimensions: head inside token inside block
  if (c.head_stride < c.head_dim || c.token_stride < c.head_stride * c.num_kv_heads ||
      c.block_stride < c.token_stride * c.block_size)
    return false;
  CUtensorMap m;
  return encode_cache_map(&m, c.k_base, c, c.block_size < kTcKeys ? c.block_size : kTcKeys);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
  const pkvd_cache& c = a.cache;
  const int G = a.num_q_heads / c.num_kv_heads;
  TcParams prm;
  const int seg_rows = c.block_size < kTcKeys ? c.block_size : kTcKeys;
  if (!encode_cache_map(&prm.tmap_k, c.k_base, c, seg_rows) || !encode_cache_map(&prm.tmap_v, c.v_base, c, seg_rows))
    return cudaErrorInvalidValue;
  prm.out = a.out;
  prm.q = a.q;
  prm.tables = a.block_tables;
  prm.max_blocks = a.max_blocks_per_seq;
  prm.num_blocks = c.num_blocks;
  prm.block_size = c.block_size;
  prm.seg_rows = seg_rows;
  prm.cu_q = a.cu_seqlens_q;
  prm.cu_k = a.cu_seqlens_k;
  prm.total_q = a.total_q;
  prm.hq = a.num_q_heads;
  prm.group = G;
  prm.tile_tokens = kTcRows / G;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.window = a.window;
  prm.err = a.err;
  const int tiles = (a.max_seqlen_q + prm.tile_tokens - 1) / prm.tile_tokens;
  prm.pairs = (tiles + 1) / 2;                                     // two Q tiles per CTA
  prm.num_seqs = a.num_seqs;
  prm.l2_bytes = device_l2_bytes();
  if (prm.pairs > 65535 || a.num_seqs > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(c.num_kv_heads, a.num_seqs, prm.pairs);
  if (c.dtype == PKVD_BF16)
    return c.head_dim == 64 ? launch_tc_typed<__nv_bfloat16, 64>(prm, grid, stream)
                            : launch_tc_typed<__nv_bfloat16, 128>(prm, grid, stream);
  return c.head_dim == 64 ? launch_tc_typed<__half, 64>(prm, grid, stream)
                          : launch_tc_typed<__half, 128>(prm, grid, stream);
}

}  // namespace pkvd
