// tree.cu -- token-tree verification with several candidates per node on
// sm_103a.
//
// The 機器之心 article "全球最強推理引擎還快2倍，斯坦福、普林斯頓破解大模型串行魔咒"
// names combining SSD with token-tree speculation as future work; the
// technical summary "超越传统SD：SSD框架全异步解码实现4.7倍平均加速" states the
// single-chain rule (accept with min(1, p/q), resample from the residual
// p_target - p_draft) that this generalises.  At a tree node, the children
// (drawn independently from the draft's q there) are tested in order against
// a target distribution r that starts as p and becomes the normalised
// residual max(0, r - q) after each rejection; an accepted child continues
// the walk, and when none is accepted the bonus is drawn from r.
//
//   k_tree_walk  one thread-block cluster of cw CTAs (512 threads) per
//                sequence.  At each visited node the two rows (target and
//                draft) are read from HBM once, split across the cluster
//                (128 blocks of 32 16-byte vectors per CTA and row, staged in
//                128 KB of shared memory by cp.async), and every
//                vocabulary-wide quantity the node needs -- the softmax
//                statistics, the residual mass after each rejection, the
//                block sums of the final draw -- is reduced from there.  Partial results meet through
//                distributed shared memory (after each cluster barrier one
//                lane per CTA copies that CTA's part, all at once) and are
//                combined in rank order by every CTA alike, so the cluster
//                takes the same decisions and its control flow stays uniform.
//                The residual after n rejections is kept in closed form,
//                max(0, p - A q) / B (see resid_w), so every element costs the
//                same whatever n is; the next node's rows (the children's)
//                are prefetched into L2 while a node is evaluated.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/ssd.h"
#include "common.cuh"

namespace {

using namespace ssd;

constexpr int kTT = 512;                     // threads per CTA
constexpr int kTWarps = kTT / 32;            // 16
constexpr int kBPW = 8;                      // blocks of 32 vectors per warp and row
constexpr int kCtaBlocks = kTWarps * kBPW;   // 128 blocks per CTA and row
constexpr int kMaxCW = 8;                    // CTAs per cluster
constexpr int kMaxNodes = 256;
constexpr int kPrefetchChildren = 8;         // children whose rows are prefetched at a node

struct TreeArgs {
  const void *target, *draft;
  int64_t seq_stride, row_stride;  // elements
  int B, N, V;
  int nvec, nfull;  // 16-byte vectors per row (the last may be partial), whole ones
  int cw;           // CTAs per cluster
  float kT;         // log2(e) / T
  int greedy;       // T == 0
  const int32_t *parent, *tokens;
  const float *u_acc, *u_bonus;
  int32_t *accept_len, *path, *bonus, *out_tokens;
  float *resid_mass;
  uint32_t *status;
};

// What a CTA contributes to one cluster-wide combination.
struct __align__(16) Part {
  float a[4];       // statistics: max and sum of p, max and sum of q; mass passes: a[0]
  uint64_t key[2];  // greedy statistics: the argmax keys of p and q
};

struct TreeSh {
  Part part[2];  // double-buffered: read by the other CTAs of the cluster
  float wred[kTWarps][4];
  uint64_t kred[kTWarps][2];
  float res[4];
  uint64_t rkey[2];
  float bsum[kCtaBlocks];  // block sums of the final draw (this CTA's blocks, in order)
  Part peer[kMaxCW];       // the cluster's parts of the current combination, copied here
  int sel[4];
  int32_t tok[kMaxNodes];
  int16_t first_child[kMaxNodes + 1];
  int16_t next_sib[kMaxNodes];
  int32_t path[kMaxNodes];
  int32_t par[kMaxNodes];
};

SSD_DEV unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
SSD_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, a multiple of 16).
SSD_DEV void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <class E>
SSD_DEV uint4 neg_inf_vector() {
  if constexpr (E::kSize == 2) return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
}

// Vector v of a row: a whole vector by one load, the partial last vector by
// element loads (-inf past V), vectors past the row as -inf.
template <class E>
SSD_DEV uint4 load_vector(const TreeArgs &a, const char *row, int v) {
  if (v < a.nfull) return __ldg(reinterpret_cast<const uint4 *>(row + static_cast<int64_t>(v) * 16));
  if (v >= a.nvec) return neg_inf_vector<E>();
  float f[E::kVec];
  const int i0 = v * E::kVec;
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) f[e] = (i0 + e < a.V) ? E::ld(row, i0 + e) : -__int_as_float(0x7f800000);
  if constexpr (E::kSize == 2) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = (__float_as_uint(f[2 * q]) >> 16) | (__float_as_uint(f[2 * q + 1]) & 0xFFFF0000u);
    return make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
}

// The distributions at the current node.  Greedy: one-hot at the argmaxes.
struct Dist {
  float kT;
  int greedy;
  float Rp, Rq;        // fl(max kT) of each row
  float invSp, invSq;  // 1 / the row sums of 2^(z kT - R)
  int ap, aq;          // greedy argmaxes
  SSD_DEV float p(float z, int idx) const {
    return greedy ? (idx == ap ? 1.f : 0.f) : __fmul_rn(ex2(__fmaf_rn(z, kT, -Rp)), invSp);
  }
  SSD_DEV float q(float z, int idx) const {
    return greedy ? (idx == aq ? 1.f : 0.f) : __fmul_rn(ex2(__fmaf_rn(z, kT, -Rq)), invSq);
  }
  // p and q of one element as a packed pair (per lane the roundings of p, q)
  SSD_DEV void pq(float zt, float zd, int idx, float &pv, float &qv) const {
    if (greedy) {
      pv = idx == ap ? 1.f : 0.f;
      qv = idx == aq ? 1.f : 0.f;
      return;
    }
    float xt, xd;
    unpack2(fma2(pack2(zt, zd), pack2(kT, kT), pack2(-Rp, -Rq)), xt, xd);
    unpack2(mul2(pack2(ex2(xt), ex2(xd)), pack2(invSp, invSq)), pv, qv);
  }
};

// The residual after n rejections at a node, r_{j+1} = max(0, r_j - q) / W_j
// from r_0 = p, in closed form: r_n = max(0, p - A_n q) / B_n with A_0 = 0,
// B_0 = 1, A_{n+1} = A_n + B_n and B_{n+1} = B_n W_n = sum_i max(0, p_i -
// A_{n+1} q_i).  (If p - A_n q > 0 then r_n - q = (p - (A_n + B_n) q) / B_n;
// otherwise both sides are 0.)  The walk keeps (A, B) and weighs element i by
// the unnormalised max(0, p_i - A q_i): O(1) per element however many
// children were rejected.
SSD_DEV float resid_w(float p, float q, float A) { return fmaxf(__fmaf_rn(-A, q, p), 0.f); }
// The bonus's weight of element idx: p before any rejection (q is then not
// computed), else the unnormalised residual.
SSD_DEV float bonus_w(const Dist &D, float zt, float zd, int idx, int n, float A) {
  if (n == 0) return D.p(zt, idx);
  float p, q;
  D.pq(zt, zd, idx, p, q);
  return resid_w(p, q, A);
}

// Thread 0 of every CTA publishes sh.part[buf]; after the cluster barrier the
// CTA copies the cw parts into its own shared memory (cluster_combine) and
// thread 0 combines them in rank order with `comb`, leaving the result in
// sh.res / sh.rkey for the CTA.
// The parts of the cluster's CTAs, copied into this CTA's shared memory.
struct Peers {
  const Part *p;
  SSD_DEV float a(int rank, int i) const { return p[rank].a[i]; }
  SSD_DEV uint64_t key(int rank, int i) const { return p[rank].key[i]; }
};

// After the cluster barrier lane r of warp 0 copies CTA r's part (32 bytes,
// two remote 16-byte loads, all CTAs at once); thread 0 then combines them.
template <class Comb>
SSD_DEV void cluster_combine(TreeSh &sh, int buf, int cw, Comb comb) {
  cluster_sync();
  if (threadIdx.x < static_cast<unsigned>(cw)) {
    uint32_t src;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(src) : "r"(smem_u32(&sh.part[buf])), "r"(threadIdx.x));
    uint4 lo, hi;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w) : "r"(src) : "memory");
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w) : "r"(src + 16) : "memory");
    uint4 *dst = reinterpret_cast<uint4 *>(&sh.peer[threadIdx.x]);
    dst[0] = lo;
    dst[1] = hi;
  }
  __syncwarp();
  if (threadIdx.x == 0) comb(Peers{sh.peer}, cw, sh);
  __syncthreads();
}

constexpr size_t kRowStage = static_cast<size_t>(kCtaBlocks) * 32 * sizeof(uint4);  // 64 KB per row

// Running totals of the CTA's block sums in block order, as one warp forms
// them: lane l sums blocks 4l .. 4l+3 in order, the lanes' totals are scanned,
// and block 4l + j's running total is the lanes-before part plus the lane's
// own run up to j.  The CTA's total is lane 31's last running total; the block
// search repeats exactly this arithmetic.
static_assert(kCtaBlocks == 4 * 32, "four block sums per lane");
SSD_DEV void block_runs(const float *bsum, int lane, float (&bs)[4], float (&run)[4], float &excl) {
#pragma unroll
  for (int j = 0; j < 4; ++j) bs[j] = bsum[4 * lane + j];
  float r[4];
  r[0] = bs[0];
#pragma unroll
  for (int j = 1; j < 4; ++j) r[j] = __fadd_rn(r[j - 1], bs[j]);
  float inc = r[3];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc = __fadd_rn(inc, t);
  }
  excl = __shfl_up_sync(0xffffffffu, inc, 1);
  if (lane == 0) excl = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) run[j] = __fadd_rn(excl, r[j]);
}

// G: T == 0 (one-hot distributions), a template argument so that the
// per-element weights carry no test of it
template <class E, bool G>
__global__ void __launch_bounds__(kTT, 1) k_tree_walk(TreeArgs a) {
  __shared__ TreeSh sh;
  extern __shared__ uint4 stage[];  // [2][kCtaBlocks * 32]: this CTA's vectors of the target, draft row
  uint4 *sT = stage, *sD = stage + kCtaBlocks * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cw = a.cw;
  const unsigned rank = cluster_rank();
  const int b = static_cast<int>(blockIdx.x) / cw;
  const int N = a.N;
  const int32_t *par = a.parent + static_cast<int64_t>(b) * N;
  uint32_t fl = 0;
  const float NEG_INF = -__int_as_float(0x7f800000);

  // children lists in index order (a node's parent must lie in [-1, m-1]),
  // built from a copy of the parents in shared memory
  for (int m = tid; m < N; m += kTT) sh.par[m] = par[m];
  for (int m = tid; m <= N; m += kTT) sh.first_child[m] = -1;
  __syncthreads();
  for (int m = tid; m < N; m += kTT) {
    const int p = sh.par[m];
    sh.tok[m] = a.tokens[static_cast<int64_t>(b) * N + m];
    sh.next_sib[m] = -1;
    if (p < -1 || p >= m) {
      fl |= kFlagBadTree;
      continue;
    }
    for (int c = m + 1; c < N; ++c) {
      if (sh.par[c] == p) {
        sh.next_sib[m] = static_cast<int16_t>(c);
        break;
      }
    }
    bool first = true;
    for (int c = p + 1; c < m && first; ++c) first = (sh.par[c] != p);
    if (first) sh.first_child[p + 1] = static_cast<int16_t>(m);
  }
  __syncthreads();

  int buf = 0, node = -1, L = 0, nrej = 0;
  float Wlast = 1.f;
  float Ar = 0.f, Br = 1.f;  // the residual at this node: max(0, p - Ar q) / Br
  Dist D;
  D.kT = a.kT;
  D.greedy = G;
  for (;;) {
    // the node's rows, into registers
    const int64_t off = static_cast<int64_t>(b) * a.seq_stride + static_cast<int64_t>(node + 1) * a.row_stride;
    const char *rowT = static_cast<const char *>(a.target) + off * E::kSize;
    const char *rowD = static_cast<const char *>(a.draft) + off * E::kSize;
    __syncthreads();  // the previous node's vectors are no longer read
#pragma unroll
    for (int k = 0; k < kBPW; ++k) {
      const int v = 32 * (static_cast<int>(rank) * kCtaBlocks + warp + kTWarps * k) + lane;
      const int i = (warp + kTWarps * k) * 32 + lane;
      if (v < a.nfull) {
        cp_async16(&sT[i], rowT + static_cast<int64_t>(v) * 16);
        cp_async16(&sD[i], rowD + static_cast<int64_t>(v) * 16);
      } else {
        sT[i] = load_vector<E>(a, rowT, v);
        sD[i] = load_vector<E>(a, rowD, v);
      }
    }
    cp_async_wait_all();
    __syncthreads();
    // the next node is one of this node's children: their rows (this CTA's
    // slices, the first kPrefetchChildren children) start moving into L2
    // while the node is evaluated
    if (tid == 0) {
      const int64_t v0 = static_cast<int64_t>(rank) * kCtaBlocks * 32;
      const int64_t v1 = min(v0 + kCtaBlocks * 32, static_cast<int64_t>(a.nfull));
      int c = sh.first_child[node + 1];
      for (int n = 0; n < kPrefetchChildren && c >= 0 && v1 > v0; ++n, c = sh.next_sib[c]) {
        const int64_t coff = (static_cast<int64_t>(b) * a.seq_stride + static_cast<int64_t>(c + 1) * a.row_stride) * E::kSize;
        prefetch_l2(static_cast<const char *>(a.target) + coff + v0 * 16, static_cast<uint32_t>((v1 - v0) * 16));
        prefetch_l2(static_cast<const char *>(a.draft) + coff + v0 * 16, static_cast<uint32_t>((v1 - v0) * 16));
      }
    }
    // statistics of p and q
    if (G) {
      uint64_t kp = 0, kq = 0;
#pragma unroll 1
      for (int k = 0; k < kBPW; ++k) {
        float ft[E::kVec], fd[E::kVec];
        E::unpack(sT[(warp + kTWarps * k) * 32 + lane], ft);
        E::unpack(sD[(warp + kTWarps * k) * 32 + lane], fd);
        const int i0 = (32 * (static_cast<int>(rank) * kCtaBlocks + warp + kTWarps * k) + lane) * E::kVec;
#pragma unroll
        for (int e = 0; e < E::kVec; ++e) {
          if (i0 + e < a.V) {
            const uint64_t ck = cand_key(ft[e], i0 + e), dk = cand_key(fd[e], i0 + e);
            kp = ck > kp ? ck : kp;
            kq = dk > kq ? dk : kq;
          }
        }
      }
      kp = warp_max_u64(kp);
      kq = warp_max_u64(kq);
      if (lane == 0) {
        sh.kred[warp][0] = kp;
        sh.kred[warp][1] = kq;
      }
      __syncthreads();
      if (tid == 0) {
        uint64_t mp = 0, mq = 0;
        for (int w = 0; w < kTWarps; ++w) {
          mp = sh.kred[w][0] > mp ? sh.kred[w][0] : mp;
          mq = sh.kred[w][1] > mq ? sh.kred[w][1] : mq;
        }
        sh.part[buf].key[0] = mp;
        sh.part[buf].key[1] = mq;
      }
      cluster_combine(sh, buf, cw, [](const Peers &all, int n, TreeSh &s) {
        uint64_t mp = 0, mq = 0;
        for (int r = 0; r < n; ++r) {
          mp = all.key(r, 0) > mp ? all.key(r, 0) : mp;
          mq = all.key(r, 1) > mq ? all.key(r, 1) : mq;
        }
        s.rkey[0] = mp;
        s.rkey[1] = mq;
      });
      D.ap = static_cast<int>(~static_cast<uint32_t>(sh.rkey[0]));
      D.aq = static_cast<int>(~static_cast<uint32_t>(sh.rkey[1]));
      D.Rp = D.Rq = 0.f;
      D.invSp = D.invSq = 1.f;
    } else {
      float mt = NEG_INF, md = NEG_INF;
#pragma unroll 1
      for (int k = 0; k < kBPW; ++k) {
        float ft[E::kVec], fd[E::kVec];
        E::unpack(sT[(warp + kTWarps * k) * 32 + lane], ft);
        E::unpack(sD[(warp + kTWarps * k) * 32 + lane], fd);
#pragma unroll
        for (int e = 0; e < E::kVec; ++e) {
          mt = fmaxf(mt, ft[e]);
          md = fmaxf(md, fd[e]);
        }
      }
      mt = ord2f(__reduce_max_sync(0xffffffffu, f2ord(mt)));
      md = ord2f(__reduce_max_sync(0xffffffffu, f2ord(md)));
      const float Rt = __fmul_rn(mt, a.kT), Rd = __fmul_rn(md, a.kT);
      float st = 0.f, sd = 0.f;
      if (mt != NEG_INF || md != NEG_INF) {
#pragma unroll 1
        for (int k = 0; k < kBPW; ++k) {
          float ft[E::kVec], fd[E::kVec];
          E::unpack(sT[(warp + kTWarps * k) * 32 + lane], ft);
          E::unpack(sD[(warp + kTWarps * k) * 32 + lane], fd);
#pragma unroll
          for (int e = 0; e < E::kVec; ++e) {
            // both rows' terms as one packed pair; a row without a finite
            // maximum adds +0
            float xt, xd;
            unpack2(fma2(pack2(ft[e], fd[e]), pack2(a.kT, a.kT), pack2(-Rt, -Rd)), xt, xd);
            const float et = mt != NEG_INF ? ex2(xt) : 0.f, ed = md != NEG_INF ? ex2(xd) : 0.f;
            unpack2(add2(pack2(st, sd), pack2(et, ed)), st, sd);
          }
        }
      }
      st = warp_sum(st);
      sd = warp_sum(sd);
      if (lane == 0) {
        sh.wred[warp][0] = mt;
        sh.wred[warp][1] = st;
        sh.wred[warp][2] = md;
        sh.wred[warp][3] = sd;
      }
      __syncthreads();
      if (tid == 0) {
        float r[4];
        for (int h = 0; h < 2; ++h) {
          float M = NEG_INF;
          for (int w = 0; w < kTWarps; ++w) M = fmaxf(M, sh.wred[w][2 * h]);
          float S = 0.f;
          if (M != NEG_INF) {
            const float R = __fmul_rn(M, a.kT);
            for (int w = 0; w < kTWarps; ++w)
              if (sh.wred[w][2 * h] != NEG_INF)
                S = __fadd_rn(S, __fmul_rn(sh.wred[w][2 * h + 1], ex2(__fsub_rn(__fmul_rn(sh.wred[w][2 * h], a.kT), R))));
          }
          r[2 * h] = M;
          r[2 * h + 1] = S;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) sh.part[buf].a[i] = r[i];
      }
      const float kT = a.kT;
      cluster_combine(sh, buf, cw, [kT, NEG_INF](const Peers &all, int n, TreeSh &s) {
        for (int h = 0; h < 2; ++h) {
          float M = NEG_INF;
          for (int r = 0; r < n; ++r) M = fmaxf(M, all.a(r, 2 * h));
          float S = 0.f;
          const float R = __fmul_rn(M, kT);
          for (int r = 0; r < n; ++r)
            if (all.a(r, 2 * h) != NEG_INF)
              S = __fadd_rn(S, __fmul_rn(all.a(r, 2 * h + 1), ex2(__fsub_rn(__fmul_rn(all.a(r, 2 * h), kT), R))));
          s.res[2 * h] = R;
          s.res[2 * h + 1] = S;
        }
      });
      D.Rp = sh.res[0];
      D.invSp = __frcp_rn(sh.res[1]);
      D.Rq = sh.res[2];
      D.invSq = __frcp_rn(sh.res[3]);
    }
    buf ^= 1;

    // the children, in index order
    nrej = 0;
    Wlast = 1.f;
    Ar = 0.f;
    Br = 1.f;
    int next = -1;
    for (int c = sh.first_child[node + 1]; c >= 0; c = sh.next_sib[c]) {
      const int x = sh.tok[c];
      if (x < 0 || x >= a.V) {
        fl |= kFlagBadToken;
        continue;
      }
      const float px = D.p(E::ld(rowT, x), x), qx = D.q(E::ld(rowD, x), x);
      // accept iff u q < r(x) = max(0, p - A q) / B
      const float rx = resid_w(px, qx, Ar);
      if (__fmul_rn(__fmul_rn(a.u_acc[static_cast<int64_t>(b) * N + c], qx), Br) < rx) {
        next = c;
        break;
      }
      // rejected: B W = sum over the row of max(0, p - (A + B) q)
      const float An = __fadd_rn(Ar, Br);
      float s = 0.f;
#pragma unroll 1
      for (int k = 0; k < kBPW; ++k) {
        float ft[E::kVec], fd[E::kVec];
        E::unpack(sT[(warp + kTWarps * k) * 32 + lane], ft);
        E::unpack(sD[(warp + kTWarps * k) * 32 + lane], fd);
        const int i0 = (32 * (static_cast<int>(rank) * kCtaBlocks + warp + kTWarps * k) + lane) * E::kVec;
#pragma unroll
        for (int e = 0; e < E::kVec; ++e) {
          float p, q;
          D.pq(ft[e], fd[e], i0 + e, p, q);
          s = __fadd_rn(s, resid_w(p, q, An));
        }
      }
      s = warp_sum(s);
      if (lane == 0) sh.wred[warp][0] = s;
      __syncthreads();
      if (tid == 0) {
        float S = 0.f;
        for (int w = 0; w < kTWarps; ++w) S = __fadd_rn(S, sh.wred[w][0]);
        sh.part[buf].a[0] = S;
      }
      cluster_combine(sh, buf, cw, [](const Peers &all, int n, TreeSh &st) {
        float S = 0.f;
        for (int r = 0; r < n; ++r) S = __fadd_rn(S, all.a(r, 0));
        st.res[0] = S;
      });
      buf ^= 1;
      const float BW = sh.res[0];
      if (BW > 0.f) {
        ++nrej;
        Wlast = __fdiv_rn(BW, Br);
        Ar = An;
        Br = BW;
      } else {
        fl |= kFlagZeroResidual;
      }
    }
    if (next >= 0) {
      if (tid == 0) sh.path[L] = next;
      ++L;
      node = next;
      continue;
    }
    break;
  }

  // the bonus: inverse CDF over r (nrej residual steps) in vocabulary order
  for (int attempt = 0; attempt < 2; ++attempt) {
#pragma unroll 1
    for (int k = 0; k < kBPW; ++k) {
      float ft[E::kVec], fd[E::kVec];
      E::unpack(sT[(warp + kTWarps * k) * 32 + lane], ft);
      E::unpack(sD[(warp + kTWarps * k) * 32 + lane], fd);
      const int i0 = (32 * (static_cast<int>(rank) * kCtaBlocks + warp + kTWarps * k) + lane) * E::kVec;
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) s = __fadd_rn(s, bonus_w(D, ft[e], fd[e], i0 + e, nrej, Ar));
      // the block total by the scan the element search repeats
      float inc = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc = __fadd_rn(inc, t);
      }
      if (lane == 31) sh.bsum[warp + kTWarps * k] = inc;
    }
    __syncthreads();
    if (warp == 0) {
      float bs[4], run[4], excl;
      block_runs(sh.bsum, lane, bs, run, excl);
      if (lane == 31) sh.part[buf].a[0] = run[3];
    }
    const float ub = a.u_bonus[b];
    cluster_combine(sh, buf, cw, [ub](const Peers &all, int n, TreeSh &st) {
      float S = 0.f;
      for (int r = 0; r < n; ++r) S = __fadd_rn(S, all.a(r, 0));
      // the CTA whose running total first exceeds u S (else the last with mass)
      const float t = __fmul_rn(ub, S);
      float run = 0.f, before = 0.f;
      int pick = -1, last = -1;
      float before_last = 0.f;
      for (int r = 0; r < n; ++r) {
        const float nx = __fadd_rn(run, all.a(r, 0));
        if (all.a(r, 0) > 0.f) {
          if (pick < 0 && nx > t) {
            pick = r;
            before = run;
          }
          last = r;
          before_last = run;
        }
        run = nx;
      }
      if (pick < 0) {
        pick = last;
        before = before_last;
      }
      st.res[0] = S;
      st.res[1] = __fsub_rn(t, before);  // the target within the chosen CTA
      st.sel[0] = pick;
    });
    buf ^= 1;
    const float S = sh.res[0];
    if (!(S > 0.f) && nrej == 0) {  // a row without any mass: no bonus
      if (rank == 0 && tid == 0) {
        a.bonus[b] = -1;
        if (a.out_tokens) a.out_tokens[static_cast<int64_t>(b) * (N + 1) + L] = -1;
      }
      break;
    }
    if (S > 0.f) {
      // the chosen CTA locates the block, its owning warp the lane and element
      if (sh.sel[0] == static_cast<int>(rank)) {
        if (warp == 0) {
          // the first block with mass whose running total exceeds t, else the last with mass
          const float t = sh.res[1];
          float bs[4], run[4], excl;
          block_runs(sh.bsum, lane, bs, run, excl);
          int pick = -1, last = -1;
          float before = 0.f, before_last = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float bef = j == 0 ? excl : run[j - 1];
            if (bs[j] > 0.f) {
              if (pick < 0 && run[j] > t) {
                pick = 4 * lane + j;
                before = bef;
              }
              last = 4 * lane + j;
              before_last = bef;
            }
          }
          const unsigned hitl = __ballot_sync(0xffffffffu, pick >= 0);
          const unsigned posl = __ballot_sync(0xffffffffu, last >= 0);
          const int src = hitl ? __ffs(hitl) - 1 : (posl ? 31 - __clz(posl) : -1);
          if (src >= 0 && lane == src) {
            sh.sel[1] = hitl ? pick : last;
            sh.res[2] = __fsub_rn(t, hitl ? before : before_last);
          } else if (src < 0 && lane == 0) {
            sh.sel[1] = -1;
            sh.res[2] = 0.f;
          }
        }
        __syncthreads();
        const int g = sh.sel[1];
        if (g >= 0 && warp == g % kTWarps) {
          // the lanes' sums of block g again, with the arithmetic of the pass
          const int i0 = (32 * (static_cast<int>(rank) * kCtaBlocks + g) + lane) * E::kVec;
          float ft[E::kVec], fd[E::kVec];
          E::unpack(sT[g * 32 + lane], ft);
          E::unpack(sD[g * 32 + lane], fd);
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < E::kVec; ++e) s = __fadd_rn(s, bonus_w(D, ft[e], fd[e], i0 + e, nrej, Ar));
          float inc = s;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float t2 = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc = __fadd_rn(inc, t2);
          }
          const float t = sh.res[2];
          float excl = __shfl_up_sync(0xffffffffu, inc, 1);
          if (lane == 0) excl = 0.f;
          const unsigned hit = __ballot_sync(0xffffffffu, s > 0.f && inc > t);
          const unsigned pos = __ballot_sync(0xffffffffu, s > 0.f);
          const int ln = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
          if (lane == ln) {
            const float tl = __fsub_rn(t, excl);
            float c = 0.f;
            int tokb = -1, lastpos = -1;
#pragma unroll
            for (int e = 0; e < E::kVec; ++e) {
              const float we = bonus_w(D, ft[e], fd[e], i0 + e, nrej, Ar);
              c = __fadd_rn(c, we);
              if (we > 0.f) {
                if (tokb < 0 && c > tl) tokb = i0 + e;
                lastpos = i0 + e;
              }
            }
            if (tokb < 0) tokb = lastpos;
            a.bonus[b] = tokb;
            if (a.out_tokens) a.out_tokens[static_cast<int64_t>(b) * (N + 1) + L] = tokb;
          }
        }
      }
      break;
    }
    // the residual lost its mass to rounding: draw from p instead
    fl |= kFlagZeroResidual;
    nrej = 0;
    Wlast = 1.f;
    Ar = 0.f;
    Br = 1.f;
  }

  if (rank == 0) {
    for (int m = tid; m < N; m += kTT) {
      a.path[static_cast<int64_t>(b) * N + m] = m < L ? sh.path[m] : -1;
      if (a.out_tokens) {
        if (m < L) a.out_tokens[static_cast<int64_t>(b) * (N + 1) + m] = sh.tok[sh.path[m]];
        else if (m > L) a.out_tokens[static_cast<int64_t>(b) * (N + 1) + m] = -1;
      }
    }
    if (a.out_tokens && tid == 0 && L < N) a.out_tokens[static_cast<int64_t>(b) * (N + 1) + N] = -1;
    if (tid == 0) {
      a.accept_len[b] = L;
      if (a.resid_mass) a.resid_mass[b] = Wlast;
    }
  }
  if (fl) atomicOr(a.status, fl);
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class E>
cudaError_t launch_tree(const TreeArgs &a, cudaStream_t s) {
  void (*kern)(TreeArgs) = a.greedy ? k_tree_walk<E, true> : k_tree_walk<E, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(2 * kRowStage));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B) * static_cast<unsigned>(a.cw));
  cfg.blockDim = dim3(kTT);
  cfg.dynamicSmemBytes = 2 * kRowStage;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.cw);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

extern "C" ssd_status_t ssd_tree_verify(const void *target, const void *draft, ssd_dtype_t dt,
                                        int64_t seq_stride, int64_t row_stride, int B, int N, int V,
                                        float T, const int32_t *parent, const int32_t *tokens,
                                        const float *u_acc, const float *u_bonus, int32_t *accept_len,
                                        int32_t *path, int32_t *bonus, int32_t *out_tokens,
                                        float *resid_mass, uint32_t *status, ssd_stream_t s) {
  if (B < 0 || N < 0 || V < 1 || (dt != SSD_F32 && dt != SSD_BF16) || !(T >= 0.f) || !isfinite(T))
    return SSD_ERR_INVALID_ARG;
  if (N > kMaxNodes) return SSD_ERR_UNSUPPORTED;
  const int es = dt == SSD_F32 ? 4 : 2;
  const long long nvec = (static_cast<long long>(V) * es + 15) / 16;
  const long long nblk = (nvec + 31) / 32;
  const long long cw = (nblk + kCtaBlocks - 1) / kCtaBlocks;
  if (cw > kMaxCW) return SSD_ERR_UNSUPPORTED;
  if (B == 0) return SSD_OK;
  if (!target || !draft || !u_bonus || !accept_len || !bonus || !status) return SSD_ERR_INVALID_ARG;
  if (N > 0 && (!parent || !tokens || !u_acc || !path)) return SSD_ERR_INVALID_ARG;
  if (seq_stride < 0 || row_stride < V) return SSD_ERR_INVALID_ARG;
  if (!aligned16(target) || !aligned16(draft) || (seq_stride * es) % 16 || (row_stride * es) % 16)
    return SSD_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * cw > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
  TreeArgs a{};
  a.target = target;
  a.draft = draft;
  a.seq_stride = seq_stride;
  a.row_stride = row_stride;
  a.B = B;
  a.N = N;
  a.V = V;
  a.nvec = static_cast<int>(nvec);
  a.nfull = static_cast<int>((static_cast<long long>(V) * es) / 16);
  a.cw = static_cast<int>(cw);
  a.greedy = (T == 0.f);
  a.kT = a.greedy ? 0.f : static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  a.parent = parent;
  a.tokens = tokens;
  a.u_acc = u_acc;
  a.u_bonus = u_bonus;
  a.accept_len = accept_len;
  a.path = path;
  a.bonus = bonus;
  a.out_tokens = out_tokens;
  a.resid_mass = resid_mass;
  a.status = status;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  const cudaError_t e = dt == SSD_F32 ? launch_tree<EF32>(a, cs) : launch_tree<EBF16>(a, cs);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
