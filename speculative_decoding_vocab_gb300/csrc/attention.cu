// attention.cu -- tree-masked decode attention over a paged bf16 KV cache on
// the sm_103a tensor cores (tcgen05 + TMEM + TMA), so the draft decodes every
// branch of the speculation tree in one forward pass: the "custom sparse
// attention mask" of the technical summary "超越传统SD：SSD框架全异步解码实现
// 4.7倍平均加速", section "工程优化与系统表现".
//
// Row i of head h (query node m = N - Nq + i) sees every prefix position and
// the tree nodes on m's ancestor-or-self path; node n's K/V sits at logical
// position prefix_len + n.  GQA: head h reads KV head h / (Hq / Hkv), and all
// the query heads of one KV head share the rows of a row tile, so each K/V page
// is read once per (sequence, KV head, row tile); at d = 64 the two row tiles of
// a KV head run in one CTA, and the second read comes from L2.
//
// A work item = (sequence b, KV head, tile of 128 query rows, range of keys).
// At d = 64 one CTA runs two independent pipelines, each on its own work item
// with 256 TMEM columns, so an SM carries two tile streams without relying on
// two CTAs being co-resident (the CUDA occupancy calculator counts one for a
// kernel that allocates TMEM).  At d = 128 it runs one, with all of shared
// memory for its K/V ring (Q and P held as 64-row tiles when at most 64 query
// rows share a KV head).
// Each pipeline is warp-specialised:
//   * a producer warp fetches the K and V pages of each 64-key tile by TMA
//     through the block table into a ring of stages (mbarrier completion);
//   * an MMA warp (one thread) issues S = Q K^T for tile t + 1 into a second
//     TMEM buffer while the softmax works on tile t, then O += P V for tile t;
//   * one softmax warpgroup per row tile (one thread per row) reads its S row
//     from TMEM, applies the tree mask and an online softmax in the log2 domain
//     (the running maximum only moves, and O is rescaled in TMEM, when it grows
//     by more than 2^8), writes P (bf16) to shared memory;
//   * the softmax threads end by normalising O, or write (O, m, l) partials that
//     a combine kernel merges when the keys are split across work items.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <cmath>

#include "../../include/ssd.h"
#include "common.cuh"

namespace ssd {

constexpr int kPage = 16;
constexpr int kMaxNodes = 128;
constexpr int kRows = 128;                  // query rows per row tile (MMA M)
constexpr int kKeys = 64;                   // keys per tile (MMA N of S, K of P V)
constexpr int kTilePages = kKeys / kPage;   // 4

// ---------------------------------------------------------------------------
// tcgen05 / TMA wrappers
// ---------------------------------------------------------------------------
SSD_DEV void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
SSD_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;"); }
SSD_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
SSD_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SSD_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc], one 128 x N x 16 step
SSD_DEV void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// arrive on `bar` once every tcgen05 op this thread issued before has completed
SSD_DEV void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane
SSD_DEV void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// The same load without its wait: both halves of a 64-column row are issued
// before tmem_wait32 (which orders every use of the registers after the wait).
SSD_DEV void tmem_ld32_async(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
SSD_DEV void tmem_wait32(uint32_t *r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
SSD_DEV void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (load, then store back)
SSD_DEV void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
SSD_DEV void tmem_st16(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

SSD_DEV void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand tile:
// start address, leading-dimension byte offset (stride between 64-element
// column blocks of an MN-major operand; unused for K-major), stride byte offset
// (between 8-row groups: 1024 B), descriptor version 1, swizzle mode 128B.
SSD_DEV uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;  // version
  d |= static_cast<uint64_t>(2u) << 61;  // SWIZZLE_128B
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128, N.
__host__ __device__ constexpr uint32_t idesc_bf16(int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(kRows >> 4) << 24);
}

// byte offset of (row r, 16-byte chunk c) inside a [rows x 128 B] SW128 block
SSD_DEV uint32_t sw128(int r, int c) { return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4); }

SSD_DEV float bf2f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }
SSD_DEV uint32_t pack_bf16x2(float lo, float hi) {
  // round to nearest even (finite inputs)
  uint32_t a = __float_as_uint(lo), b = __float_as_uint(hi);
  a += 0x7FFFu + ((a >> 16) & 1u);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (a >> 16) | (b & 0xFFFF0000u);
}
SSD_DEV float bf16_round(float x) {
  uint32_t a = __float_as_uint(x);
  a += 0x7FFFu + ((a >> 16) & 1u);
  return __uint_as_float(a & 0xFFFF0000u);
}

SSD_DEV void mbar_arrive1(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// two fp32 -> bf16x2 (round to nearest even): lo in the low half
SSD_DEV uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// 64 bits of the 128-bit node mask starting at bit `off` (bits below 0 read 0)
SSD_DEV uint64_t mask_bits(const uint32_t *w, int off) {
  uint64_t r = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int sh = 32 * k - off;  // position of word k relative to the window
    const uint64_t x = w[k];
    if (sh >= 0 && sh < 64) r |= x << sh;
    else if (sh < 0 && sh > -32) r |= x >> (-sh);
  }
  return r;
}

struct AttnArgs {
  const uint16_t *q;
  const int32_t *table;
  int maxb;
  int64_t num_blocks;
  const int32_t *prefix_len, *parent;
  int B, N, Nq, Hq, Hkv, group, nrows, mtiles, splits, tiles_per_split;
  int items;     // work items: (sequence, KV head) x row-tile groups x key splits
  float scale_log2;  // scale * log2(e)
  uint16_t *out;
  float *lse;
  float *part_o;   // [B*Hkv][mtiles][splits][128][d] fp32 (splits > 1)
  float *part_ml;  // [B*Hkv][mtiles][splits][128][3]
  uint32_t *status;
};

// Shared-memory plan of a CTA at head dimension D that runs PL independent
// pipelines (each its own work item, Q, K/V ring, barriers and TMEM columns),
// each with MT row tiles of which RA rows of Q and P are held in shared
// memory.  PL = 2 puts two tile streams on an SM within one CTA.  RA < 128
// serves problems with at most RA query rows: the MMA still reads 128 rows of
// A, and rows RA..127 fall on the next buffer (finite or not, they only feed
// TMEM lanes that no thread reads).
// NPB P buffers per row tile: with two, the softmax writes P of tile t while
// P V of tile t - 1 runs; with one, it first waits for that P V.
template <int D, int MT, int PL, int RA = kRows, int NPB = 2>
struct AttnCfg {
  static_assert(RA == kRows || (MT == 1 && RA % 32 == 0 && RA < kRows), "trimmed row tiles: one per pipeline");
  static constexpr int kQBytes = RA * D * 2;         // one row tile of Q
  static constexpr int kKVBytes = kKeys * D * 2;     // K or V of one key tile
  static constexpr int kPBytes = RA * kKeys * 2;     // one P buffer of one row tile
  static constexpr int kFixed = MT * kQBytes + MT * NPB * kPBytes;
  static constexpr int kStagesFit = (216 * 1024 / PL - kFixed) / (2 * kKVBytes);
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  // TMEM: S buffers (MT x 2 x 64 columns), then O (MT x D); a power of two
  static constexpr uint32_t kOCol = MT * 2 * kKeys;
  static constexpr uint32_t kTmemNeed = kOCol + MT * D;
  static constexpr uint32_t kTmemCols = kTmemNeed <= 128 ? 128 : (kTmemNeed <= 256 ? 256 : 512);
  static_assert(kTmemCols * PL <= 512, "TMEM of the pipelines");
  static constexpr int kQ = 0;
  static constexpr int kP = kQ + MT * kQBytes;
  static constexpr int kKV = kP + MT * NPB * kPBytes;
  static constexpr int kPipe = kKV + kStages * 2 * kKVBytes;  // one pipeline's region
  static constexpr int kTable = PL * kPipe;  // then each pipeline's block-table entries
  static constexpr int kPWarps = 4 * MT + 2;  // warps of one pipeline
  static constexpr int kPThreads = kPWarps * 32;
  static constexpr int kThreads = PL * kPThreads;
  static constexpr int kTmaWarp = 4 * MT, kMmaWarp = 4 * MT + 1;  // within a pipeline
  static_assert(kStages >= 2, "at least two K/V stages");
  static_assert(kPipe % 1024 == 0, "each pipeline's swizzled tiles stay 1024-byte aligned");
  static_assert(PL == 1 || MT == 1, "two pipelines hold one row tile each");
  // the 128 A rows the MMA reads from the last Q column block and the last P
  // buffer stay inside the pipeline's region
  static_assert(kQ + MT * kQBytes - RA * 128 + kRows * 128 <= kPipe, "Q rows read by the MMA");
  static_assert(kP + (MT * NPB - 1) * kPBytes + kRows * 128 <= kPipe, "P rows read by the MMA");
  static_assert(NPB == 1 || NPB == 2, "one or two P buffers");
};

// int entries of one pipeline's block-table slice (16-byte multiple)
__host__ __device__ inline int attn_tab_stride(int tiles_per_split) { return (tiles_per_split * kTilePages + 3) & ~3; }

// LX: the exact row sums are kept (the log-sum-exp output); without it only
// the sums of the bf16 P that normalise O are.
template <int D, int MT, int PL, int RA, int NPB, bool LX>
__global__ void __launch_bounds__(AttnCfg<D, MT, PL, RA, NPB>::kThreads, 1)
    k_branch_attn_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ AttnArgs a) {
  using CF = AttnCfg<D, MT, PL, RA, NPB>;
  constexpr int NS = CF::kStages;
  constexpr bool kEarlyExp = PL == 1;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  uint8_t *const smem_all =
      reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t kv_full_[PL][NS], kv_empty_[PL][NS];
  __shared__ __align__(8) uint64_t s_full_[PL][MT][2], s_free_[PL][MT][2], p_full_[PL][MT][2], pv_done_[PL][MT][2];
  __shared__ uint32_t tmem_base;
  __shared__ uint32_t anc_[PL][kMaxNodes][kMaxNodes / 32];
  __shared__ int par_[PL][kMaxNodes];
  __shared__ volatile int s_abort_[PL];

  // This thread's pipeline, and its warp and thread numbers within it.  The
  // softmax warpgroups come first (a warp reaches the TMEM lanes 32 (w % 4) ..
  // + 31 by its warp number w in the CTA), then each pipeline's producer and
  // MMA warps.
  constexpr int kSoftWarps = 4 * MT;
  const int gw = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool soft_w = gw < PL * kSoftWarps;
  const int pl = soft_w ? gw / kSoftWarps : (gw - PL * kSoftWarps) / 2;
  const int warp = soft_w ? gw % kSoftWarps : kSoftWarps + (gw - PL * kSoftWarps) % 2;
  const int tid = warp * 32 + lane;
  uint64_t(&kv_full)[NS] = kv_full_[pl];
  uint64_t(&kv_empty)[NS] = kv_empty_[pl];
  uint64_t(&s_full)[MT][2] = s_full_[pl];
  uint64_t(&s_free)[MT][2] = s_free_[pl];
  uint64_t(&p_full)[MT][2] = p_full_[pl];
  uint64_t(&pv_done)[MT][2] = pv_done_[pl];
  uint32_t(&anc)[kMaxNodes][kMaxNodes / 32] = anc_[pl];
  int(&par)[kMaxNodes] = par_[pl];
  volatile int &s_abort = s_abort_[pl];
  uint8_t *const smem = smem_all + pl * CF::kPipe;
  // the pipeline's work item: (sequence, KV head), group of row tiles, key range
  const int mgroups = (a.mtiles + MT - 1) / MT;
  const int item = blockIdx.x * PL + pl;
  const bool has_item = item < a.items;
  const int it = has_item ? item : 0;
  const int split = it % a.splits, mg = (it / a.splits) % mgroups, bh = it / (a.splits * mgroups);
  const int b = bh / a.Hkv, hk = bh % a.Hkv;
  const int N = a.N;
  const int L_in = a.prefix_len[b];
  const int L = max(0, L_in);
  const int nkeys = L + N;
  const int ntiles_all = (nkeys + kKeys - 1) / kKeys;
  const int t_begin = split * a.tiles_per_split;
  const int t_end = min(ntiles_all, t_begin + a.tiles_per_split);
  const int nt = has_item ? max(0, t_end - t_begin) : 0;
  const int mt_here = has_item ? min(MT, a.mtiles - mg * MT) : 0;  // row tiles of this pipeline
  const float NEG_INF = -__int_as_float(0x7f800000);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int m = 0; m < MT; ++m) {
      // softmax warps of row tile m that hold a valid row (the others sit out)
      const int rows_m = a.nrows - (mg * MT + m) * kRows;
      const int nact = rows_m <= 0 ? 1 : min(4, (min(rows_m, kRows) + 31) / 32);
      for (int u = 0; u < 2; ++u) {
        mbar_init(&s_full[m][u], 1);
        mbar_init(&s_free[m][u], nact);
        mbar_init(&p_full[m][u], nact);
        mbar_init(&pv_done[m][u], 1);
      }
    }
    fence_mbar_init();
    s_abort = 0;
    // a prefix the block table cannot hold: the keys past it stay hidden
    if (has_item && (L_in < 0 || nkeys > a.maxb * kPage)) atomicOr(a.status, kFlagBadPrefix);
  }
  if (pl == 0 && warp == CF::kMmaWarp) {
    tmem_alloc(&tmem_base, PL * CF::kTmemCols);
    tmem_relinquish();
  }
  // the tree's parent indices (one coalesced load), then the ancestor-or-self
  // masks walked in shared memory
  for (int m = tid; m < N; m += CF::kPThreads) par[m] = a.parent[static_cast<int64_t>(b) * N + m];
  __syncthreads();
  for (int m = tid; m < N; m += CF::kPThreads) {
    uint32_t bits[kMaxNodes / 32] = {0, 0, 0, 0};
    int x = m;
    bool bad = false;
    while (x >= 0) {
      bits[x >> 5] |= 1u << (x & 31);
      const int px = par[x];
      if (px < -1 || px >= x) {
        bad = true;
        break;
      }
      x = px;
    }
    if (bad) atomicOr(a.status, kFlagBadTree);
#pragma unroll
    for (int w = 0; w < kMaxNodes / 32; ++w) anc[m][w] = bits[w];
  }
  // block-table entries of this pipeline's key range (-1: past the table or the keys, or a bad id)
  int *tab = reinterpret_cast<int *>(smem_all + CF::kTable) + pl * attn_tab_stride(a.tiles_per_split);
  const int page0 = t_begin * kTilePages;
  const int npages = nt * kTilePages;
  for (int i = tid; i < npages; i += CF::kPThreads) {
    const int lp = page0 + i;
    int blk = -1;
    if (lp < a.maxb && lp * kPage < nkeys) {
      blk = a.table[static_cast<int64_t>(b) * a.maxb + lp];
      if (blk < 0 || blk >= a.num_blocks) {
        atomicOr(a.status, kFlagBadBlock);
        blk = -1;
      }
    }
    tab[i] = blk;
  }
  // Q tiles: each softmax thread stages its row, 128-byte swizzled, in d/64 column blocks
  const int m_own = warp >> 2;                        // softmax warps: row tile
  const int r_own = (warp & 3) * 32 + lane;           // row within the tile (= TMEM lane)
  const int row = (mg * MT + m_own) * kRows + r_own;  // row within (b, hk)
  const bool softmax_thread = warp < 4 * MT;
  const bool row_valid = softmax_thread && m_own < mt_here && row < a.nrows;
  const int qi = row_valid ? row / a.group : 0;
  const int head = hk * a.group + (row_valid ? row % a.group : 0);
  // a softmax warp without a valid row sits the loop out; its P rows stay zero
  const bool warp_active = __any_sync(0xffffffffu, row_valid);
  if (softmax_thread && !warp_active && r_own < RA) {
#pragma unroll
    for (int u = 0; u < NPB; ++u)
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        *reinterpret_cast<uint4 *>(smem + CF::kP + (m_own * NPB + u) * CF::kPBytes + sw128(r_own, q4)) =
            make_uint4(0, 0, 0, 0);
  }
  if (softmax_thread && r_own < RA) {
    const uint16_t *qrow = a.q + ((static_cast<int64_t>(b) * a.Nq + qi) * a.Hq + head) * D;
    uint8_t *qt = smem + CF::kQ + m_own * CF::kQBytes;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row_valid) v = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
      *reinterpret_cast<uint4 *>(qt + (c >> 3) * (RA * 128) + sw128(r_own, c & 7)) = v;
    }
  }
  fence_proxy_async();  // generic-proxy writes of Q -> visible to the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base + pl * CF::kTmemCols;  // this pipeline's columns
  int issued = 0;  // producer: tiles whose copies were issued

  if (warp == CF::kTmaWarp) {
    // ---------------- producer: K and V pages of each tile into the ring; lane 0
    // takes the stage, one lane per page and operand issues its copy
    constexpr int kCopies = 2 * kTilePages * (D / 64);
    for (int i = 0; i < nt; ++i) {
      const int st = i % NS;
      int ok = 1;
      if (lane == 0) {
        if (s_abort) ok = 0;
        else if (i >= NS && !mbar_wait_sleep(&kv_empty[st], ((i / NS) - 1) & 1)) {
          s_abort = 1;
          ok = 0;
        }
        if (ok) mbar_arrive_expect_tx(&kv_full[st], 2 * kTilePages * (D / 64) * (kPage * 128));
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane < kCopies) {
        const int p = lane / (2 * (D / 64)), r = lane % (2 * (D / 64));
        const int kv = r & 1, h = r >> 1;
        const int blk = tab[i * kTilePages + p];
        // pages past the keys or with a bad id load block 0 (finite values, masked out)
        const int y = ((blk >= 0 ? blk : 0) * a.Hkv + hk) * kPage;
        uint8_t *dst = smem + CF::kKV + (st * 2 + kv) * CF::kKVBytes + h * (kKeys * 128) + p * (kPage * 128);
        tma_load_2d(dst, kv ? &vmap : &kmap, h * 64, y, &kv_full[st]);
      }
      issued = i + 1;
    }
  } else if (warp == CF::kMmaWarp) {
    // ---------------- MMA issue (one thread): S(t) then O += P(t-1) V(t-1)
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(kKeys, 0);
      const uint32_t idesc_o = idesc_bf16(D, 1);
      auto issue_pv = [&](int u) {
        const int st = u % NS;
        const uint32_t v_base = smem_u32(smem + CF::kKV + st * 2 * CF::kKVBytes + CF::kKVBytes);
        for (int m = 0; m < mt_here; ++m) {
          if (!mbar_wait_sleep(&p_full[m][u & 1], (u >> 1) & 1)) {
            s_abort = 1;
            return;
          }
          tc_fence_after();
          const uint32_t p_base = smem_u32(smem + CF::kP + (m * NPB + u % NPB) * CF::kPBytes);
          const uint32_t tO = tmem + CF::kOCol + m * D;
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            // P: 16 keys = 32 bytes of each 128-byte row; V: 16 keys = two 8-key groups of 1024 B,
            // d blocks of 64 columns kKeys * 128 B apart
            umma_bf16(tO, smem_desc_sw128(p_base + kk * 32, 16), smem_desc_sw128(v_base + kk * 2048, kKeys * 128),
                      idesc_o, (u > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&pv_done[m][u & 1]);
        }
        umma_commit(&kv_empty[st]);
      };
      for (int i = 0; i < nt && !s_abort; ++i) {
        const int st = i % NS;
        if (!mbar_wait_sleep(&kv_full[st], (i / NS) & 1)) {
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t k_base = smem_u32(smem + CF::kKV + st * 2 * CF::kKVBytes);
        for (int m = 0; m < mt_here; ++m) {
          if (i >= 2 && !mbar_wait_sleep(&s_free[m][i & 1], ((i - 2) >> 1) & 1)) {
            s_abort = 1;
            break;
          }
          tc_fence_after();
          const uint32_t q_base = smem_u32(smem + CF::kQ + m * CF::kQBytes);
          const uint32_t tS = tmem + (m * 2 + (i & 1)) * kKeys;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qoff = (kk >> 2) * (RA * 128) + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * (kKeys * 128) + (kk & 3) * 32;
            umma_bf16(tS, smem_desc_sw128(q_base + qoff, 16), smem_desc_sw128(k_base + koff, 16), idesc_s,
                      kk > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[m][i & 1]);
        }
        if (s_abort) break;
        if (i >= 1) issue_pv(i - 1);
      }
      if (nt >= 1 && !s_abort) issue_pv(nt - 1);
    }
  } else if (m_own < mt_here && warp_active) {
    // ---------------- softmax: one thread per row of row tile m_own
    const int m = m_own;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t my_anc[kMaxNodes / 32] = {0, 0, 0, 0};
    if (row_valid) {
      const int node = N - a.Nq + qi;
#pragma unroll
      for (int w = 0; w < kMaxNodes / 32; ++w) my_anc[w] = anc[node][w];
    }
    const float c = a.scale_log2;
    float m_used = NEG_INF;
    uint64_t l2 = pack2(0.f, 0.f), lx2 = pack2(0.f, 0.f);  // sums of the bf16 P (normalises O) and exact (lse)
    for (int i = 0; i < nt; ++i) {
      const int t = t_begin + i, u = i & 1;
      if (!__all_sync(0xffffffffu, !s_abort && mbar_wait_sleep(&s_full[m][u], (i >> 1) & 1))) {
        s_abort = 1;
        break;
      }
      tc_fence_after();
      float s[kKeys];
      {
        uint32_t rs[kKeys];
        tmem_ld32_async(tmem + (m * 2 + u) * kKeys + lane_off, rs);
        tmem_ld32_async(tmem + (m * 2 + u) * kKeys + 32 + lane_off, rs + 32);
        tmem_wait32(rs);
        tmem_wait32(rs + 32);
#pragma unroll
        for (int j = 0; j < kKeys; ++j) s[j] = __uint_as_float(rs[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(&s_free[m][u]);
      // visibility of the tile's 64 keys for this row
      const int kbase = t * kKeys;
      uint64_t vis = ~0ull;
      bool full = kbase + kKeys <= L;
      uint32_t pmask = 0;
#pragma unroll
      for (int p = 0; p < kTilePages; ++p) pmask |= (tab[i * kTilePages + p] >= 0 ? 1u : 0u) << p;
      full = full && pmask == 0xFu;
      if (!full) {
        const uint64_t pre = (L - kbase >= kKeys) ? ~0ull : (L > kbase ? ((1ull << (L - kbase)) - 1ull) : 0ull);
        const uint64_t tree = mask_bits(my_anc, kbase - L) & ~pre;
        uint64_t pg = 0;
#pragma unroll
        for (int p = 0; p < kTilePages; ++p)
          if ((pmask >> p) & 1u) pg |= 0xFFFFull << (16 * p);
        const uint64_t inr = (nkeys - kbase >= kKeys) ? ~0ull : ((1ull << (nkeys - kbase)) - 1ull);
        vis = (pre | tree) & pg & inr;
      }
      if (!full) {  // hidden keys score -inf (their P is then 0)
#pragma unroll
        for (int j = 0; j < kKeys; ++j) s[j] = ((vis >> j) & 1ull) ? s[j] : NEG_INF;
      }
      // tile maximum (eight running maxima, then a tree), scaled to log2 units
      float t8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) t8[j] = s[j];
#pragma unroll
      for (int j = 8; j < kKeys; ++j) t8[j & 7] = fmaxf(t8[j & 7], s[j]);
#pragma unroll
      for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) t8[j] = fmaxf(t8[j], t8[j + w]);
      float tmax = row_valid ? t8[0] : NEG_INF;
      tmax = (tmax == NEG_INF) ? NEG_INF : __fmul_rn(tmax, c);
      const bool grow = tmax != NEG_INF && (m_used == NEG_INF || tmax > m_used + 8.f);
      // a row whose maximum moved rescales its sums now and its O (in TMEM) below
      const bool rescale = grow && m_used != NEG_INF;
      const float f = rescale ? ex2(m_used - tmax) : 1.f;
      if (grow) {
        if (rescale) {
          l2 = fma2(l2, pack2(f, f), pack2(0.f, 0.f));
          if constexpr (LX) lx2 = fma2(lx2, pack2(f, f), pack2(0.f, 0.f));
        }
        m_used = tmax;
      }
      // the P buffer of tile i is free once P V of tile i - NPB completed; O is
      // rescaled in TMEM (after P V of tile i - 1) when a row's maximum moved
      auto wait_p_and_rescale = [&]() -> bool {
        if (i >= NPB && !__all_sync(0xffffffffu, mbar_wait_sleep(&pv_done[m][(i - NPB) & 1], ((i - NPB) >> 1) & 1)))
          return false;
        if (i >= 1 && __any_sync(0xffffffffu, rescale)) {
          if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[m][u ^ 1], ((i - 1) >> 1) & 1))) return false;
          tc_fence_after();
          float o[16];
#pragma unroll
          for (int cc = 0; cc < D / 16; ++cc) {
            const uint32_t ta = tmem + CF::kOCol + m * D + cc * 16 + lane_off;
            tmem_ld16(ta, o);
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = __fmul_rn(o[j], f);
            tmem_st16(ta, o);
          }
          tc_fence_before();
        }
        return true;
      };
      // One pipeline per CTA: the exponentials run before the wait, while P V
      // of the previous tile does.  Two pipelines per CTA (d = 64) share the
      // SM's exponential unit and are faster with the wait first.
      if (!kEarlyExp && !wait_p_and_rescale()) {
        s_abort = 1;
        break;
      }
      // P = 2^(s c - m) in bf16, in registers
      const uint64_t c2 = pack2(c, c), nm2 = pack2(-m_used, -m_used);
      const bool any = row_valid && m_used != NEG_INF;
      uint64_t la[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)}, lxa[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)};
      uint32_t pk[kKeys / 2];
#pragma unroll
      for (int h = 0; h < kKeys / 2; ++h) {
        const int j = 2 * h;
        float p0 = 0.f, p1 = 0.f;
        if (any) {
          float x0, x1;
          unpack2(fma2(pack2(s[j], s[j + 1]), c2, nm2), x0, x1);
          p0 = ex2(x0);
          p1 = ex2(x1);
        }
        const uint32_t pb = cvt_bf16x2(p0, p1);
        if constexpr (LX) lxa[h & 1] = add2(lxa[h & 1], pack2(p0, p1));
        la[h & 1] = add2(la[h & 1], pack2(__uint_as_float(pb << 16), __uint_as_float(pb & 0xFFFF0000u)));
        pk[h] = pb;
      }
      l2 = add2(l2, add2(la[0], la[1]));
      if constexpr (LX) lx2 = add2(lx2, add2(lxa[0], lxa[1]));
      if (kEarlyExp && !wait_p_and_rescale()) {
        s_abort = 1;
        break;
      }
      // 128 bytes of this row in the swizzled K-major P tile
      uint8_t *prow = smem + CF::kP + (m * NPB + i % NPB) * CF::kPBytes;
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        *reinterpret_cast<uint4 *>(prow + sw128(r_own, q4)) =
            make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
      fence_proxy_async();  // P (generic writes) -> visible to the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive1(&p_full[m][u]);
    }
    // ---------------- epilogue: O after the last P V
    float lo, hi;
    unpack2(l2, lo, hi);
    const float l = __fadd_rn(lo, hi);
    unpack2(lx2, lo, hi);
    const float lx = __fadd_rn(lo, hi);
    bool have = false;
    if (nt > 0 && !s_abort) {
      if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[m][(nt - 1) & 1], ((nt - 1) >> 1) & 1))) s_abort = 1;
      else have = true;
      tc_fence_after();
    }
    const int64_t orow = (static_cast<int64_t>(b) * a.Nq + qi) * a.Hq + head;
    const int mtile = mg * MT + m;
    if (have) {
      float o[32];
      if (a.splits == 1) {
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          tmem_ld32(tmem + CF::kOCol + m * D + cc * 32 + lane_off, o);
          if (row_valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + orow * D + cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[q4] = make_uint4(pack_bf16x2(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv),
                                   pack_bf16x2(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv),
                                   pack_bf16x2(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv),
                                   pack_bf16x2(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv));
          }
        }
        if (row_valid && a.lse) a.lse[orow] = (lx > 0.f) ? (m_used + log2f(lx)) * 0.69314718055994531f : NEG_INF;
      } else {
        const size_t pidx = ((static_cast<size_t>(bh) * a.mtiles + mtile) * a.splits + split) * kRows + r_own;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          tmem_ld32(tmem + CF::kOCol + m * D + cc * 32 + lane_off, o);
          float4 *dst = reinterpret_cast<float4 *>(a.part_o + pidx * D + cc * 32);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) dst[q4] = make_float4(o[q4 * 4], o[q4 * 4 + 1], o[q4 * 4 + 2], o[q4 * 4 + 3]);
        }
        a.part_ml[pidx * 3 + 0] = m_used;
        a.part_ml[pidx * 3 + 1] = l;
        a.part_ml[pidx * 3 + 2] = lx;
      }
    } else if (!s_abort && a.splits > 1) {
      // no key of this split: an empty partial
      const size_t pidx = ((static_cast<size_t>(bh) * a.mtiles + mtile) * a.splits + split) * kRows + r_own;
      a.part_ml[pidx * 3 + 0] = NEG_INF;
      a.part_ml[pidx * 3 + 1] = 0.f;
      a.part_ml[pidx * 3 + 2] = 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s_abort && tid == 0) atomicOr(a.status, kFlagWaitTimeout);
  if (warp == CF::kTmaWarp && lane == 0 && s_abort) {
    // copies still in flight land before the CTA's shared memory is released
    for (int i = max(0, issued - NS); i < issued; ++i) (void)mbar_wait(&kv_full[i % NS], (i / NS) & 1);
  }
  if (pl == 0 && warp == CF::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, PL * CF::kTmemCols);
  }
}

// Merge the key-split partials of every (sequence, query row, head).
template <int D>
__global__ void __launch_bounds__(128) k_attn_combine(const AttnArgs a) {
  const int bh = blockIdx.x, b = bh / a.Hkv, hk = bh % a.Hkv;
  const int mt = blockIdx.y;
  const int tid = threadIdx.x;
  const int row = mt * kRows + tid;
  if (row >= a.nrows) return;
  const int qi = row / a.group, head = hk * a.group + row % a.group;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const size_t base = ((static_cast<size_t>(bh) * a.mtiles + mt) * a.splits) * kRows + tid;
  float M = NEG_INF;
  for (int s = 0; s < a.splits; ++s) M = fmaxf(M, a.part_ml[(base + s * kRows) * 3]);
  float Lsum = 0.f, Lx = 0.f;
  float acc[D];
#pragma unroll
  for (int e = 0; e < D; ++e) acc[e] = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const size_t p = base + s * kRows;
    const float m = a.part_ml[p * 3], l = a.part_ml[p * 3 + 1], lx = a.part_ml[p * 3 + 2];
    if (m == NEG_INF || l == 0.f) continue;
    const float f = ex2(m - M);
    Lsum += l * f;
    Lx += lx * f;
    const float4 *src = reinterpret_cast<const float4 *>(a.part_o + p * D);
#pragma unroll
    for (int e = 0; e < D / 4; ++e) {
      const float4 x = src[e];
      acc[4 * e] += x.x * f;
      acc[4 * e + 1] += x.y * f;
      acc[4 * e + 2] += x.z * f;
      acc[4 * e + 3] += x.w * f;
    }
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  const int64_t orow = (static_cast<int64_t>(b) * a.Nq + qi) * a.Hq + head;
  uint32_t *dst = reinterpret_cast<uint32_t *>(a.out + orow * D);
#pragma unroll
  for (int e = 0; e < D / 2; ++e) dst[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  if (a.lse) a.lse[orow] = Lx > 0.f ? (M + log2f(Lx)) * 0.69314718055994531f : NEG_INF;
}

}  // namespace ssd

using namespace ssd;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D view of a paged cache: [num_blocks * Hkv * 16 rows, d], boxes of 16 rows x 64 elements
bool make_kv_map(CUtensorMap *m, const void *base, int64_t num_blocks, int Hkv, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(num_blocks) * Hkv * kPage};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[2] = {64, kPage};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int attn_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// At d = 128, problems with at most this many query rows per KV head hold
// 64-row Q and one 64-row P buffer, which leaves shared memory for six K/V
// stages instead of four.
constexpr int kTrimRows = 64;

struct AttnPlan {
  int nrows, mtiles, pipes, splits, tiles_per_split;
  size_t part_o_bytes, part_ml_bytes;
};

// One row tile per work item; two pipelines per CTA at d = 64 (the two row
// tiles of a KV head then read its pages once from HBM), one at d = 128 (all
// of shared memory for the K/V ring), one CTA per SM.  Keys are split so that
// the work items fill whole waves of pipelines, with at least 4 tiles per
// split.
AttnPlan plan_attention(int B, int Nq, int Hq, int Hkv, int d, int max_keys) {
  AttnPlan p;
  p.nrows = (Hq / Hkv) * Nq;
  p.mtiles = (p.nrows + kRows - 1) / kRows;
  p.pipes = d == 64 ? 2 : 1;
  const int ntiles = (max_keys + kKeys - 1) / kKeys;
  const long base = static_cast<long>(B) * Hkv * p.mtiles;
  const long slots = static_cast<long>(attn_num_sms()) * p.pipes;  // concurrent work items
  // estimated time in tile-steps: whole waves x (tiles per split + a work
  // item's set-up, about kSetupTiles tiles: masks, Q, TMEM, the first copies)
  constexpr double kSetupTiles = 4.0;
  int best = 1;
  double best_cost = 0.0;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && ntiles / s < 4) break;
    const long items = base * s;
    const double waves = std::ceil(static_cast<double>(items) / slots);
    const double cost = waves * (std::ceil(static_cast<double>(ntiles) / s) + kSetupTiles);
    if (s == 1 || cost < best_cost * 0.97) {
      best_cost = cost;
      best = s;
    }
  }
  p.splits = best;
  p.tiles_per_split = (ntiles + best - 1) / best;
  if (p.tiles_per_split < 1) p.tiles_per_split = 1;
  const size_t nparts = best > 1 ? static_cast<size_t>(B) * Hkv * p.mtiles * best * kRows : 0;
  p.part_o_bytes = nparts * d * sizeof(float);
  p.part_ml_bytes = nparts * 3 * sizeof(float);
  return p;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

template <int D, int MT, int PL, int RA = kRows, int NPB = 2>
int attention_smem(const AttnArgs &a) {
  using CF = AttnCfg<D, MT, PL, RA, NPB>;
  return CF::kTable + PL * attn_tab_stride(a.tiles_per_split) * 4 + 1024;
}

// Whether the configuration's dynamic + static shared memory for this key
// range fits the per-block opt-in limit.
template <int D, int MT, int PL, int RA = kRows, int NPB = 2>
bool attention_fits(const AttnArgs &a) {
  static const int room = [] {
    cudaFuncAttributes fa;
    int dev = 0, optin = 0;
    if (cudaFuncGetAttributes(&fa, k_branch_attn_tc<D, MT, PL, RA, NPB, true>) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return 227 * 1024 - 4096;
    return optin - static_cast<int>(fa.sharedSizeBytes);
  }();
  return attention_smem<D, MT, PL, RA, NPB>(a) <= room;
}

template <int D, int MT, int PL, int RA = kRows, int NPB = 2>
cudaError_t launch_attention(const CUtensorMap &kmap, const CUtensorMap &vmap, const AttnArgs &a,
                             cudaStream_t cs) {
  // the exact sums only when the log-sum-exp is written (at d = 64 the
  // two-pipeline kernel keeps them: measured faster with both sums)
  void (*kern)(const CUtensorMap, const CUtensorMap, const AttnArgs);
  if constexpr (D == 64)
    kern = k_branch_attn_tc<D, MT, PL, RA, NPB, true>;
  else
    kern = a.lse ? k_branch_attn_tc<D, MT, PL, RA, NPB, true> : k_branch_attn_tc<D, MT, PL, RA, NPB, false>;
  using CF = AttnCfg<D, MT, PL, RA, NPB>;
  const int smem = attention_smem<D, MT, PL, RA, NPB>(a);
  if (!attention_fits<D, MT, PL, RA, NPB>(a)) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.items + PL - 1) / PL);
  kern<<<grid, CF::kThreads, smem, cs>>>(kmap, vmap, a);
  e = cudaGetLastError();
  if (e == cudaSuccess && a.splits > 1) {
    k_attn_combine<D><<<dim3(a.B * a.Hkv, a.mtiles), 128, 0, cs>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

extern "C" {

size_t ssd_attention_workspace_size(int B, int Nq, int Hq, int Hkv, int d, int max_prefix) {
  if (B <= 0 || Nq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_prefix < 0) return 0;
  const AttnPlan p = plan_attention(B, Nq, Hq, Hkv, d, max_prefix + kMaxNodes);
  return align256(p.part_o_bytes) + align256(p.part_ml_bytes);
}

ssd_status_t ssd_branch_attention(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_table, int maxb, int64_t num_blocks,
                                  const int32_t *prefix_len, const int32_t *parent, int B, int N, int Nq, int Hq,
                                  int Hkv, int d, float scale, void *out, float *lse, uint32_t *status, void *ws,
                                  size_t ws_bytes, ssd_stream_t s) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || !(scale > 0.f) || !isfinite(scale)) return SSD_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return SSD_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SSD_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16 || N < 1 || N > kMaxNodes || Nq < 1 || Nq > N) return SSD_ERR_UNSUPPORTED;
  if (B == 0) return SSD_OK;
  if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !parent || !out || !status || maxb < 1 ||
      num_blocks < 1)
    return SSD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return SSD_ERR_UNSUPPORTED;
  // keys per sequence are bounded by the block table
  const int max_keys = maxb * kPage;
  const AttnPlan p = plan_attention(B, Nq, Hq, Hkv, d, max_keys);
  const size_t need = align256(p.part_o_bytes) + align256(p.part_ml_bytes);
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = static_cast<const uint16_t *>(q);
  a.table = block_table;
  a.maxb = maxb;
  a.num_blocks = num_blocks;
  a.prefix_len = prefix_len;
  a.parent = parent;
  a.B = B;
  a.N = N;
  a.Nq = Nq;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = Hq / Hkv;
  a.nrows = p.nrows;
  a.mtiles = p.mtiles;
  // without room for the split partials the keys are not split (documented at
  // the declaration: correct, but slower for long prefixes)
  const bool split_ok = p.splits > 1 && ws && ws_bytes >= need && !(reinterpret_cast<uintptr_t>(ws) & 255u);
  a.splits = split_ok ? p.splits : 1;
  a.tiles_per_split = split_ok ? p.tiles_per_split : (max_keys + kKeys - 1) / kKeys;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = static_cast<uint16_t *>(out);
  a.lse = lse;
  a.part_o = split_ok ? static_cast<float *>(ws) : nullptr;
  a.part_ml = split_ok ? reinterpret_cast<float *>(static_cast<char *>(ws) + align256(p.part_o_bytes)) : nullptr;
  a.status = status;
  CUtensorMap kmap, vmap;
  if (!make_kv_map(&kmap, k_cache, num_blocks, Hkv, d) || !make_kv_map(&vmap, v_cache, num_blocks, Hkv, d))
    return SSD_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  a.items = B * Hkv * p.mtiles * a.splits;
  cudaError_t e;
  if (d == 64) {
    e = launch_attention<64, 1, 2, kRows, 1>(kmap, vmap, a, cs);
  } else if (p.nrows <= kTrimRows && attention_fits<128, 1, 1, kTrimRows, 1>(a)) {
    // six stages with 64-row tiles and one P buffer
    e = launch_attention<128, 1, 1, kTrimRows, 1>(kmap, vmap, a, cs);
  } else {
    // more rows, or a key range whose block-table slice leaves no room for
    // six stages: four
    e = launch_attention<128, 1, 1>(kmap, vmap, a, cs);
  }
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
