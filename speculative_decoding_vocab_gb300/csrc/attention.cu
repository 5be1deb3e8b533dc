// attention.cu -- tree-masked decode attention over a paged bf16 KV cache on
// the sm_103a tensor cores (tcgen05 + TMEM + TMA), so the draft decodes every
// branch of the speculation tree in one forward pass: the "custom sparse
// attention mask" of the technical summary "超越传统SD：SSD框架全异步解码实现
// 4.7倍平均加速", section "工程优化与系统表现".
//
// Row i of head h (query node m = N - Nq + i) sees every prefix position and
// the tree nodes on m's ancestor-or-self path; node n's K/V sits at logical
// position prefix_len + n.  GQA: head h reads KV head h / (Hq / Hkv), and all
// the query heads of one KV head share a CTA's rows, so each K/V page is read
// once per (sequence, KV head, row tile).
//
// One CTA = (sequence b, KV head, tile of 128 query rows, range of keys):
//   * Q tile (128 x d) staged once in shared memory, 128-byte swizzled;
//   * K and V pages (16 positions x d) fetched by TMA through the block table
//     into a two-stage ring of 128-key tiles (mbarrier completion);
//   * S = Q K^T by tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in TMEM);
//   * one thread per row reads its S row from TMEM, applies the tree mask and
//     an online softmax in the log2 domain (the running max is only moved,
//     and O rescaled in TMEM, when it grows by more than 2^8), writes P (bf16)
//     to shared memory;
//   * O += P V by tcgen05.mma with V as an MN-major operand, in TMEM;
//   * the epilogue normalises O, or writes (O, m, l) partials that a combine
//     kernel merges when the keys are split across CTAs.
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
constexpr int kRows = 128;        // query rows per CTA (MMA M)
constexpr int kTiles = 2;         // K/V ring stages
// keys per tile (MMA N of S, K of P V): 128 at d = 64, 64 at d = 128, so that
// two CTAs (2 x 112 KiB of shared memory, 2 x 256 TMEM columns) share an SM
template <int D>
struct KeysPerTile {
  static constexpr int value = D == 64 ? 128 : 64;
};
constexpr int kAttnThreads = 128;  // one thread per query row
constexpr uint32_t kTmemCols = 256;  // S: keys-per-tile columns, O: d columns

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

struct AttnArgs {
  const uint16_t *q;
  const int32_t *table;
  int maxb;
  int64_t num_blocks;
  const int32_t *prefix_len, *parent;
  int B, N, Nq, Hq, Hkv, group, nrows, mtiles, splits, tiles_per_split;
  float scale_log2;  // scale * log2(e)
  uint16_t *out;
  float *lse;
  float *part_o;   // [B*Hkv][mtiles][splits][128][d] fp32 (splits > 1)
  float *part_ml;  // [B*Hkv][mtiles][splits][128][2]
  uint32_t *status;
};

template <int D>
struct AttnSmem {
  static constexpr int kKeys = KeysPerTile<D>::value;
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kKVBytes = kKeys * D * 2;  // one of K or V for a tile
  static constexpr int kPBytes = kRows * kKeys * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kV = kK + kTiles * kKVBytes;
  static constexpr int kP = kV + kTiles * kKVBytes;
  static constexpr int kTable = kP + kPBytes;  // block-table entries of the CTA's key range
  static constexpr int kTotal = kTable;        // all tile offsets multiples of 1024
};

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 2)
    k_branch_attn_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const AttnArgs a) {
  using SL = AttnSmem<D>;
  constexpr int kKeys = SL::kKeys;
  constexpr int kPages = kKeys / kPage;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kTiles];
  __shared__ __align__(8) uint64_t sdone, odone;
  __shared__ uint32_t tmem_base;
  __shared__ uint32_t anc[kMaxNodes][kMaxNodes / 32];
  __shared__ uint8_t page_ok[kTiles][1];
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int bh = blockIdx.x, b = bh / a.Hkv, hk = bh % a.Hkv;
  const int mt = blockIdx.y, split = blockIdx.z;
  const int N = a.N;
  const int L = max(0, a.prefix_len[b]);
  const int nkeys = L + N;
  const int ntiles_all = (nkeys + kKeys - 1) / kKeys;
  const int t_begin = split * a.tiles_per_split;
  const int t_end = min(ntiles_all, t_begin + a.tiles_per_split);
  const int row = mt * kRows + tid;  // this thread's query row within (b, hk)
  const bool row_valid = row < a.nrows;
  const int qi = row_valid ? row / a.group : 0;
  const int head = hk * a.group + (row_valid ? row % a.group : 0);
  const float NEG_INF = -__int_as_float(0x7f800000);

  if (tid == 0) {
    for (int s = 0; s < kTiles; ++s) mbar_init(&full[s], 1);
    mbar_init(&sdone, 1);
    mbar_init(&odone, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // ancestor-or-self masks of the tree nodes
  for (int m = tid; m < N; m += kAttnThreads) {
    uint32_t bits[kMaxNodes / 32] = {0, 0, 0, 0};
    int x = m;
    bool bad = false;
    while (x >= 0) {
      bits[x >> 5] |= 1u << (x & 31);
      const int px = a.parent[static_cast<int64_t>(b) * N + x];
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
  // block-table entries of this CTA's key range, staged once
  int *tab = reinterpret_cast<int *>(smem + SL::kTable);
  const int page0 = t_begin * kPages;
  const int npages_here = max(0, (t_end - t_begin) * kPages);
  for (int i = tid; i < npages_here; i += kAttnThreads) {
    const int lp = page0 + i;
    tab[i] = (lp < a.maxb) ? a.table[static_cast<int64_t>(b) * a.maxb + lp] : -1;
  }
  // Q tile: this thread's row, 128-byte swizzled, in d/64 column blocks
  {
    const uint16_t *qrow = a.q + ((static_cast<int64_t>(b) * a.Nq + qi) * a.Hq + head) * D;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row_valid) v = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
      *reinterpret_cast<uint4 *>(smem + SL::kQ + (c >> 3) * (kRows * 128) + sw128(tid, c & 7)) = v;
    }
  }
  fence_proxy_async();  // generic-proxy writes of Q -> visible to the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t tS = tmem;          // columns [0, 128)
  const uint32_t tO = tmem + kKeys;  // columns [kKeys, kKeys + D)
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  // producer (thread 0): fetch the K and V pages of tile t into stage s
  auto issue_tile = [&](int t, int s) {
    uint8_t ok = 0;
    const int expect = 2 * kPages * (D / 64) * (kPage * 128);
    mbar_arrive_expect_tx(&full[s], expect);
    for (int p = 0; p < kPages; ++p) {
      const int lp = t * kPages + p;  // logical page
      int blk = -1;
      if (lp * kPage < nkeys) {
        blk = tab[lp - page0];
        if (blk >= 0 && blk < a.num_blocks) ok |= static_cast<uint8_t>(1u << p);
        else atomicOr(a.status, kFlagBadBlock);
      }
      // pages past the end or with a bad id load block 0 (finite values, masked out)
      const int use = (ok >> p) & 1 ? blk : 0;
      const int y = (use * a.Hkv + hk) * kPage;
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tma_load_2d(smem + SL::kK + s * SL::kKVBytes + h * (kKeys * 128) + p * (kPage * 128), &kmap, h * 64, y,
                    &full[s]);
        tma_load_2d(smem + SL::kV + s * SL::kKVBytes + h * (kKeys * 128) + p * (kPage * 128), &vmap, h * 64, y,
                    &full[s]);
      }
    }
    page_ok[s][0] = ok;
  };

  uint32_t full_ph = 0, s_ph = 0, o_ph = 0;
  if (tid == 0) {
    for (int i = 0; i < kTiles && t_begin + i < t_end; ++i) issue_tile(t_begin + i, i);
  }
  __syncthreads();

  // this row's node mask
  uint32_t my_anc[kMaxNodes / 32] = {0, 0, 0, 0};
  if (row_valid) {
    const int node = N - a.Nq + qi;
#pragma unroll
    for (int w = 0; w < kMaxNodes / 32; ++w) my_anc[w] = anc[node][w];
  }
  float m_used = NEG_INF, l = 0.f, lx = 0.f;  // l: sum of the bf16 P (normalises O); lx: exact (lse)
  const uint32_t idesc_s = idesc_bf16(kKeys, 0);
  const uint32_t idesc_o = idesc_bf16(D, 1);
  const uint32_t q_base = smem_u32(smem + SL::kQ);
  const uint32_t p_base = smem_u32(smem + SL::kP);
  bool issued_pv = false;

  for (int t = t_begin; t < t_end; ++t) {
    const int i = t - t_begin;
    const int s = i & 1;
    // ---- S = Q K^T
    if (tid == 0) {
      bool ok = mbar_wait(&full[s], (full_ph >> s) & 1u);
      full_ph ^= 1u << s;
      if (!ok) s_abort = 1;
      else {
        tc_fence_after();
        const uint32_t k_base = smem_u32(smem + SL::kK + s * SL::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kRows * 128) + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * (kKeys * 128) + (kk & 3) * 32;
          umma_bf16(tS, smem_desc_sw128(q_base + off, 16), smem_desc_sw128(k_base + koff, 16), idesc_s, kk > 0);
        }
        umma_commit(&sdone);
      }
    }
    __syncthreads();
    if (s_abort) break;
    if (!mbar_wait(&sdone, s_ph)) s_abort = 1;
    s_ph ^= 1;
    tc_fence_after();
    __syncthreads();
    if (s_abort) break;
    const uint8_t pok = page_ok[s][0];
    // ---- pass 1: masked, scaled tile maximum of this row
    const int kbase = t * kKeys;
    float tmax = NEG_INF;
    float v[32];
#pragma unroll
    for (int c = 0; c < kKeys / 32; ++c) {
      tmem_ld32(tS + lane_off + c * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int kj = c * 32 + j;
        const int pos = kbase + kj;
        bool vis = row_valid && ((pok >> (kj >> 4)) & 1) && pos < nkeys;
        if (vis && pos >= L) {
          const int n = pos - L;
          vis = (my_anc[n >> 5] >> (n & 31)) & 1u;
        }
        if (vis) tmax = fmaxf(tmax, v[j] * a.scale_log2);
      }
    }
    float m_new = m_used;
    bool need = false;
    if (tmax != NEG_INF && (m_used == NEG_INF || tmax > m_used + 8.f)) {
      m_new = tmax;
      need = true;
    }
    // ---- PV of the previous tile must be done before O and P are touched
    if (i > 0) {
      if (!mbar_wait(&odone, o_ph)) s_abort = 1;
      o_ph ^= 1;
      tc_fence_after();
    }
    if (tid == 0 && i > 0 && t + 1 < t_end && !s_abort) issue_tile(t + 1, s ^ 1);
    // ---- rescale O rows whose running maximum moved (never before the first P V)
    if (i > 0 && __any_sync(0xffffffffu, need)) {
      const float f = need ? ex2(m_used - m_new) : 1.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(tO + lane_off + c * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= f;
        tmem_st32(tO + lane_off + c * 32, v);
      }
    }
    if (need) {
      const float f = (m_used == NEG_INF) ? 0.f : ex2(m_used - m_new);
      l *= f;
      lx *= f;
      m_used = m_new;
    }
    // ---- pass 2: P = 2^(s - m) (bf16) into shared memory, row sum
    uint8_t *prow = smem + SL::kP;
#pragma unroll
    for (int c = 0; c < kKeys / 32; ++c) {
      tmem_ld32(tS + lane_off + c * 32, v);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float pr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kj = c * 32 + j + h;
          const int pos = kbase + kj;
          bool vis = row_valid && ((pok >> (kj >> 4)) & 1) && pos < nkeys;
          if (vis && pos >= L) {
            const int n = pos - L;
            vis = (my_anc[n >> 5] >> (n & 31)) & 1u;
          }
          float p = 0.f;
          if (vis && m_used != NEG_INF) p = ex2(v[j + h] * a.scale_log2 - m_used);
          lx += p;
          p = bf16_round(p);
          l += p;
          pr[h] = p;
        }
        pk[j >> 1] = pack_bf16x2(pr[0], pr[1]);
      }
      // 32 keys = 64 bytes = 4 chunks of 16 B in key block (c >> 1)
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int chunk = (c & 1) * 4 + q4;
        *reinterpret_cast<uint4 *>(prow + (c >> 1) * (kRows * 128) + sw128(tid, chunk)) =
            make_uint4(pk[q4 * 4 + 0], pk[q4 * 4 + 1], pk[q4 * 4 + 2], pk[q4 * 4 + 3]);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (s_abort) break;
    // ---- O += P V
    if (tid == 0) {
      tc_fence_after();
      const uint32_t v_base = smem_u32(smem + SL::kV + s * SL::kKVBytes);
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk) {
        const uint32_t poff = (kk >> 2) * (kRows * 128) + (kk & 3) * 32;
        // V: 16 keys = two 8-key groups of 1024 B; d blocks of 64 at kKeys*128 B
        const uint32_t voff = kk * 2048;
        umma_bf16(tO, smem_desc_sw128(p_base + poff, 16), smem_desc_sw128(v_base + voff, kKeys * 128), idesc_o,
                  (i > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&odone);
    }
    issued_pv = true;
  }
  // ---- epilogue
  if (issued_pv) {
    if (!mbar_wait(&odone, o_ph)) s_abort = 1;
    o_ph ^= 1;
    tc_fence_after();
  }
  __syncthreads();
  const bool abort_all = s_abort != 0;
  if (abort_all && tid == 0) atomicOr(a.status, kFlagWaitTimeout);
  if (!abort_all && issued_pv) {
    float o[32];
    const int64_t orow = (static_cast<int64_t>(b) * a.Nq + qi) * a.Hq + head;
    if (a.splits == 1) {
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(tO + lane_off + c * 32, o);
        if (row_valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(a.out + orow * D + c * 32);
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
      const size_t pidx = ((static_cast<size_t>(bh) * a.mtiles + mt) * a.splits + split) * kRows + tid;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(tO + lane_off + c * 32, o);
        float4 *dst = reinterpret_cast<float4 *>(a.part_o + pidx * D + c * 32);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) dst[q4] = make_float4(o[q4 * 4], o[q4 * 4 + 1], o[q4 * 4 + 2], o[q4 * 4 + 3]);
      }
      a.part_ml[pidx * 3 + 0] = m_used;
      a.part_ml[pidx * 3 + 1] = l;
      a.part_ml[pidx * 3 + 2] = lx;
    }
  } else if (!abort_all && a.splits > 1) {
    // no key of this split: an empty partial
    const size_t pidx = ((static_cast<size_t>(bh) * a.mtiles + mt) * a.splits + split) * kRows + tid;
    a.part_ml[pidx * 3 + 0] = NEG_INF;
    a.part_ml[pidx * 3 + 1] = 0.f;
    a.part_ml[pidx * 3 + 2] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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

struct AttnPlan {
  int nrows, mtiles, splits, tiles_per_split;
  size_t part_o_bytes, part_ml_bytes;
};

// Split the keys of every (sequence, KV head, row tile) so that the CTAs fill
// whole waves of the GPU (2 resident per SM), with at least 2 tiles per split.
AttnPlan plan_attention(int B, int Nq, int Hq, int Hkv, int d, int max_keys) {
  AttnPlan p;
  const int kt = d == 64 ? KeysPerTile<64>::value : KeysPerTile<128>::value;
  p.nrows = (Hq / Hkv) * Nq;
  p.mtiles = (p.nrows + kRows - 1) / kRows;
  const int ntiles = (max_keys + kt - 1) / kt;
  const long base = static_cast<long>(B) * Hkv * p.mtiles;
  const long slots = 2L * attn_num_sms();
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 8; ++s) {
    if (s > 1 && ntiles / s < 2) break;
    const long ctas = base * s;
    const double waves = static_cast<double>(ctas) / slots;
    const double eff = waves / std::ceil(waves);
    if (eff > best_eff + 0.03) {
      best_eff = eff;
      best = s;
    }
  }
  p.splits = best;
  p.tiles_per_split = (ntiles + best - 1) / best;
  if (p.tiles_per_split < 1) p.tiles_per_split = 1;
  const size_t nparts = best > 1 ? static_cast<size_t>(base) * best * kRows : 0;
  p.part_o_bytes = nparts * d * sizeof(float);
  p.part_ml_bytes = nparts * 3 * sizeof(float);
  return p;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

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
  if (p.splits > 1 && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))) {
    // not enough workspace for split partials: run unsplit
  }
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
  const bool split_ok = p.splits > 1 && ws && ws_bytes >= need && !(reinterpret_cast<uintptr_t>(ws) & 255u);
  a.splits = split_ok ? p.splits : 1;
  const int kt = d == 64 ? KeysPerTile<64>::value : KeysPerTile<128>::value;
  a.tiles_per_split = split_ok ? p.tiles_per_split : (max_keys + kt - 1) / kt;
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
  dim3 grid(B * Hkv, a.mtiles, a.splits);
  cudaError_t e;
  if (d == 64) {
    const int smem = AttnSmem<64>::kTotal + a.tiles_per_split * (KeysPerTile<64>::value / kPage) * 4 + 1024;
    e = cudaFuncSetAttribute(k_branch_attn_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) {
      k_branch_attn_tc<64><<<grid, kAttnThreads, smem, cs>>>(kmap, vmap, a);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess && a.splits > 1) {
      k_attn_combine<64><<<dim3(B * Hkv, a.mtiles), 128, 0, cs>>>(a);
      e = cudaGetLastError();
    }
  } else {
    const int smem = AttnSmem<128>::kTotal + a.tiles_per_split * (KeysPerTile<128>::value / kPage) * 4 + 1024;
    e = cudaFuncSetAttribute(k_branch_attn_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) {
      k_branch_attn_tc<128><<<grid, kAttnThreads, smem, cs>>>(kmap, vmap, a);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess && a.splits > 1) {
      k_attn_combine<128><<<dim3(B * Hkv, a.mtiles), 128, 0, cs>>>(a);
      e = cudaGetLastError();
    }
  }
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
