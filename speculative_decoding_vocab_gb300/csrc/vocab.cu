// vocab.cu -- the vocabulary-wide kernels of one speculation round on sm_103a:
// Saguaro draft sampling, lossless verification with the residual / bonus
// draw, outcome prediction (top-F_k guesses), the speculation-cache lookup and
// the exact analytics of a round.
//
// Method: speculative-speculative decoding with the Saguaro algorithm as the
// 機器之心 article "全球最強推理引擎還快2倍，斯坦福、普林斯頓破解大模型串行魔咒"
// (section "SSD 如何實現草擬與驗證并行？") and the technical summary
// "超越传统SD：SSD框架全异步解码实现4.7倍平均加速" (sections "投机解码的瓶颈与 SSD 的
// 核心机制" and "Saguaro 算法" parts 1-2) describe it; the readings of the
// missing formulas are stated in include/ssd.h at each call.
//
// Structure: a vocabulary call is up to three kernels, chained by
// programmatic dependent launches (each may start while the previous one
// drains and waits for its completion with griddepcontrol.wait):
//   k_stats  the HBM pass, which carries nearly all of the call's bytes.  Each
//            warp reduces one segment of a logit row (256 16-byte vectors,
//            eight blocks of 32) held in registers: its maximum, the sum of
//            2^(z log2e/T - fl(max log2e/T)), its argmax where it is used,
//            and, for rows a draw reads, the eight block sums; for draft rows
//            with a top-F list, the eight block maximum keys.  No barrier and
//            no shared memory: a CTA is four independent warps (eight CTAs per
//            SM, so the grid's last wave is small).
//   k_pair   one CTA per row pair (target row j, draft row j) of a sequence:
//            merges the segment records into row statistics, selects the
//            top-F from the block maxima (re-reading the few candidate blocks,
//            from L2), draws d_{j+1} from the Saguaro weights (segment, block,
//            then one block read again), takes p(d), q'(d) and the position's
//            verdict; at position K+1 it draws the bonus for full acceptance.
//   k_resid  (verification at T > 0) units of 16 KiB of each row, or of up to
//            eight times that when the batch is large (one wave of units): the
//            sequence's first rejected pair read again (from L2) for the block sums of
//            max(0, p - q'); the unit with the sequence's last ticket draws the
//            bonus from them and writes the outputs and the cache lookup.  A
//            sequence that needs no residual is finished by its first unit.
//            The analytics call runs the units over every pair for the sums of
//            min(p, q') and max(0, p - q').
// In a verification call k_pair publishes each pair's record (and its guess
// list) through ready words in the workspace -- with C = 1 or T = 0 before the
// top-F selection, which the record then does not depend on -- and k_resid
// units wait only for their own sequence's records instead of the whole pair
// grid.  ssd_round_pipelined launches k_stats as a dependent of the previous
// call's k_resid, so the next batch's HBM pass overlaps this verification tail.
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/ssd.h"
#include "common.cuh"

namespace ssd {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSegVec = 256;                   // 16-byte vectors per segment (one warp)
constexpr int kSegBlocks = 8;                  // blocks of 32 vectors per segment
constexpr int kUnitSeg = kWarps;               // segments per residual-unit staging (k_resid)
constexpr int kStatWarps = 4;                  // segments (one per warp) per k_stats CTA: 128 threads,
                                               // 8 CTAs per SM, a fine-grained last wave
constexpr int kResSeg = kWarps / 2;            // segments per group of a residual unit (two warps per segment)
constexpr int kMaxSeg = 1024;                  // rows of at most 4 MiB
constexpr int kMaxSub = 8;                     // groups of kResSeg segments per residual unit (<= 32 segments)
constexpr int kMaxUnits = kMaxSeg / kResSeg;   // 256
constexpr int kMaxK = 16;
constexpr int kMaxSlots = 2 * (kMaxK + 1);
constexpr int kMaxF = 256;
constexpr int kCandCap = 512;
constexpr int kNone = 0x7fffffff;
constexpr int kTgt = 0, kDft = 1;
// A draw whose target lies within kNearTie * W of an edge of the chosen
// element's bin, and an acceptance test with |u - p/q'| < kNearTie, is a
// near-tie: fp32 and exact arithmetic may decide it differently.  Such
// events are counted (the optional near_ties output).
constexpr float kNearTie = 1e-6f;

// A pair's record and its guess list are published by writing kReady into
// the pair's two ready words (release); k_resid polls its sequence's words
// (acquire) instead of waiting for the whole pair grid.  The sequence's last
// residual unit sets them back to 0 once the pair grid has completed, so every
// verification call leaves them 0; a 64-bit value makes a match in a never
// used workspace practically impossible.
constexpr unsigned long long kReady = 0x9E3779B97F4A7C15ull;
constexpr uint32_t kReadyPolls = 1u << 16;  // then the grid's completion is awaited instead

// flag bits of a position's record
constexpr uint32_t kRecAccepted = 1u;   // the acceptance test passed
constexpr uint32_t kRecDrawNear = 2u;   // the draw of d was a near-tie
constexpr uint32_t kRecBonusNear = 4u;  // the bonus draw after full acceptance was a near-tie
constexpr uint32_t kRecZero = 8u;       // greedy: the residual has no mass

struct __align__(16) SegRec {
  float m;  // segment maximum
  float s;  // sum over the segment of 2^(z kT - fl(m kT)) (0 when greedy)
  int a;    // lowest index holding m (argmax rows), else the segment's first index
  float t;  // rows a draw reads: the total of the eight block sums by warp_runs' arithmetic
};
// What k_pair leaves for k_resid about position j+1 (row pair j).
struct __align__(16) PairRec {
  int d;          // draft token d_{j+1}
  float p, q;     // p_j(d), q'_j(d) (p < 0: d outside [0, V))
  uint32_t fl;    // kRec* bits
  int bt;         // bonus after full acceptance (position K+1); greedy: the bonus at every position
  float W;        // greedy: the residual's mass; analytics: W_j
  float N;        // Saguaro normaliser 1 - (1 - C) sum_S q
  float hp;       // analytics: the guesses' target probability
  uint64_t keyF;  // the smallest key of S (0: S empty)
  float hr;       // analytics: the guesses' residual probability
  float al;       // analytics: alpha_j
  float gm[2];    // target / draft row maximum
  float gs[2];    // target / draft sum of 2^(z kT - fl(gm kT))
};
static_assert(sizeof(PairRec) == 64, "records are copied as four 16-byte pieces");
struct RowSlot {
  int16_t tensor;  // 0 target, 1 draft
  int16_t row;
  uint8_t keys;    // block maximum keys (draft rows with a top-F list)
  uint8_t blocks;  // block sums (rows a draw reads)
  uint8_t arg;     // argmax tracked (greedy rows and top-1 lists)
  uint8_t pad;
};

struct VocabArgs {
  const void *target, *draft;
  int64_t seq_stride, row_stride;  // elements
  int B, K, V;
  int nvec, nfull;  // 16-byte vectors per row (the last may be partial), whole ones
  int nseg, nblk, nunits;
  int unit_sub;  // groups of kResSeg segments per residual unit (1 .. kMaxSub)
  int nslots, npairs;
  int b0;  // k_stats: first sequence of this launch (grid z = sequence - b0)
  float kT;    // log2(e) / T
  int greedy;  // T == 0
  float C;
  int do_sample, do_verify, do_predict, do_lookup, do_analytics;
  RowSlot slot[kMaxSlots];
  int tsl[kMaxK + 1], dsl[kMaxK + 1];  // slot of target / draft row j (-1: not read)
  int F[kMaxK + 1];                    // fan-out F_j
  int Fs[kMaxK + 1];                   // top-F list built for draft row j (F_j or 0)
  int foff[kMaxK + 2];
  // workspace
  uint32_t *ctr;   // [0] sequences finished, [1] hits, [2 + b] sequence tickets, [2 + B + b K + j] analytics pair tickets
  SegRec *seg;     // [B][nslots][nseg]
  float *bsum;     // [B][nslots][nblk]
  uint32_t *bkey;  // [B][nslots][nblk]
  PairRec *rec;    // [B][K+1]
  float2 *umass;   // residual units: [B][nunits] masses of max(0, p - q') and of p
  float2 *useg;    // residual segment masses: [B][nseg]
  float2 *amass;   // analytics units: [B][K][nunits] sums of min(p, q') and max(0, p - q')
  // inputs / outputs
  const float *u_draft, *u_acc, *u_bonus;
  const int32_t *d_in;
  const int32_t *payload;
  int32_t *d_out;
  float *qd_out;
  int32_t *fill_payload;  // cache fill: the draw of sequence b also goes to fill_payload[b * fill_stride + fill_col]
  unsigned long long *ready;  // verification: [B][K+1][2] record / guess list published (kReady), else 0; NULL otherwise
  int pipelined;              // host: k_stats may start while the previous kernel on the stream still runs
  int fill_stride, fill_col;
  int32_t *accept_len, *out_tokens, *bonus;
  float *accept_prob, *resid_mass;
  int32_t *guess;
  float *guess_q;
  int32_t *slot_out, *next_tokens;
  uint32_t *hits;
  uint32_t *near_ties;
  float *an_alpha, *an_resid_w, *an_p_accept, *an_hit_mass, *an_hit_rate, *an_exp_tokens;
  uint32_t *status;
  unsigned long long *trace;     // optional: 8 words per CTA (see ssd_set_trace)
  long trace_pair, trace_resid;  // first trace entry of k_pair's and of k_resid's CTAs
};

SSD_DEV const char *row_ptr(const VocabArgs &a, int tensor, int b, int row, int esize) {
  const char *base = reinterpret_cast<const char *>(tensor ? a.draft : a.target);
  return base + (static_cast<int64_t>(b) * a.seq_stride + static_cast<int64_t>(row) * a.row_stride) * esize;
}
SSD_DEV size_t slot_index(const VocabArgs &a, int b, int slot) { return static_cast<size_t>(b) * a.nslots + slot; }

// Publishing a pair's results (release) and waiting for them (acquire, bounded).
SSD_DEV void publish_ready(unsigned long long *p) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(kReady) : "memory");
}
SSD_DEV bool wait_ready(const unsigned long long *p) {
  for (uint32_t it = 0; it < kReadyPolls; ++it) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    if (v == kReady) return true;
    __nanosleep(64);
  }
  return false;
}

// Trace marks (ssd_set_trace): %globaltimer.
SSD_DEV unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// A statistics CTA's entry: identity and start mark (the other words stay 0).
SSD_DEV void trace_start(const VocabArgs &a, long idx, int b, int j) {
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  unsigned long long *tr = a.trace + 8 * idx;
  tr[0] = (static_cast<unsigned long long>(smid) << 48) | (static_cast<unsigned long long>(b & 0xFFFFF) << 20) |
          static_cast<unsigned long long>(j & 0xFFFFF);
  tr[1] = now_ns();
#pragma unroll
  for (int k = 2; k < 8; ++k) tr[k] = 0ull;
}
SSD_DEV void trace_entry(const VocabArgs &a, long idx, int kind, int b, int j, const unsigned long long *mk) {
  if (!a.trace || threadIdx.x != 0) return;
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  unsigned long long *tr = a.trace + 8 * idx;
  tr[0] = (static_cast<unsigned long long>(smid) << 48) | (static_cast<unsigned long long>(kind) << 40) |
          (static_cast<unsigned long long>(b & 0xFFFFF) << 20) | static_cast<unsigned long long>(j & 0xFFFFF);
#pragma unroll
  for (int k = 1; k < 8; ++k) tr[k] = mk[k];
}

// ---------------------------------------------------------------------------
// vectors, weights and fixed-order sums
// ---------------------------------------------------------------------------
template <class E>
SSD_DEV uint4 neg_inf_vec() {
  const uint32_t w = (E::kSize == 2) ? 0xFF80FF80u : 0xFF800000u;
  return make_uint4(w, w, w, w);
}
// One 16-byte vector of a row that is streamed once (no L1 allocation).
SSD_DEV uint4 ld_stream(const char *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
// Vector v of a row: a whole vector by one load, the partial last vector by
// element loads (-inf past V), vectors past the row as -inf.
template <class E>
SSD_DEV uint4 row_vec(const VocabArgs &a, const char *row, int v) {
  if (v < a.nfull) return __ldg(reinterpret_cast<const uint4 *>(row + static_cast<int64_t>(v) * 16));
  if (v >= a.nvec) return neg_inf_vec<E>();
  float f[E::kVec];
  const int i0 = v * E::kVec;
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) f[e] = (i0 + e < a.V) ? E::ld(row, i0 + e) : -__int_as_float(0x7f800000);
  uint32_t w[4];
  if constexpr (E::kSize == 2) {
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = (__float_as_uint(f[2 * q]) >> 16) | (__float_as_uint(f[2 * q + 1]) & 0xFFFF0000u);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = __float_as_uint(f[q]);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <class E>
SSD_DEV float vec_max(const uint4 &w) {
  if constexpr (E::kSize == 2) {
    const uint32_t t = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
    return fmaxf(__uint_as_float(t << 16), __uint_as_float(t & 0xFFFF0000u));
  } else {
    return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
  }
}
// The lane sum of a vector's weights, with one fixed association used by
// every pass and every draw: even and odd elements summed separately in order
// (a packed add), then the two.
template <int N>
SSD_DEV float lane_sum(const float *x) {
  uint64_t acc = pack2(x[0], x[1]);
#pragma unroll
  for (int h = 1; h < N / 2; ++h) acc = add2(acc, pack2(x[2 * h], x[2 * h + 1]));
  float lo, hi;
  unpack2(acc, lo, hi);
  return __fadd_rn(lo, hi);
}
// A block's running weight: lane sums combined by a Hillis-Steele inclusive
// scan over the warp.
SSD_DEV float warp_incl_scan(float x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = __fadd_rn(x, t);
  }
  return x;
}
// The eight block sums of a warp: pr[k] is this lane's part of block k.
// Recursive halving (partners 16, 8, 4 lanes apart keep half of the blocks
// each), then a butterfly over the last four lanes of a block.  Lane l ends
// with the sum of block l / 4.
SSD_DEV float warp_block_sums(const float (&pr)[kSegBlocks]) {
  const int lane = threadIdx.x & 31;
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float q4[4], q2[2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float keep = b4 ? pr[4 + k] : pr[k], send = b4 ? pr[k] : pr[4 + k];
    q4[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float keep = b3 ? q4[2 + k] : q4[k], send = b3 ? q4[k] : q4[2 + k];
    q2[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  float q = __fadd_rn(b2 ? q2[1] : q2[0], __shfl_xor_sync(0xffffffffu, b2 ? q2[0] : q2[1], 4));
  q = __fadd_rn(q, __shfl_xor_sync(0xffffffffu, q, 2));
  q = __fadd_rn(q, __shfl_xor_sync(0xffffffffu, q, 1));
  return q;
}
// Cumulative masses, one warp: lane l sums its run of `per` consecutive
// masses in order, the runs are combined by a Hillis-Steele inclusive scan.
// Returns the lane's exclusive prefix; *W = the total (every lane).
SSD_DEV float warp_runs(const float *mass, int n, int per, float *W) {
  const int lane = threadIdx.x & 31;
  float run = 0.f;
  for (int k = 0, i = lane * per; k < per && i < n; ++k, ++i) run = __fadd_rn(run, mass[i]);
  const float incl = warp_incl_scan(run);
  *W = __shfl_sync(0xffffffffu, incl, 31);
  const float ex = __shfl_up_sync(0xffffffffu, incl, 1);
  return lane == 0 ? 0.f : ex;
}
// The total of n masses with the arithmetic of warp_runs (one warp; every
// lane returns it).
SSD_DEV float warp_total(const float *mass, int n) {
  float W;
  (void)warp_runs(mass, n, (n + 31) / 32, &W);
  return W;
}
// One warp: the first of n masses whose running sum (warp_runs) exceeds the
// target (u * total, or u itself when u_is_target) with positive mass; when
// rounding leaves the target past the end, the last positive mass (*fb set).
// Returns its index (-1 when the total is 0) and, in every lane, *rem = the
// target minus the mass before it and *W = the total.
SSD_DEV int warp_locate(const float *mass, int n, float u, bool u_is_target, float *rem, float *Wout, bool *fb) {
  const int lane = threadIdx.x & 31;
  const int per = (n + 31) / 32;
  float W;
  float cum = warp_runs(mass, n, per, &W);
  const float target = u_is_target ? u : __fmul_rn(u, W);
  int hit = -1, lpos = -1;
  float hb = 0.f, lb = 0.f;
  for (int k = 0, i = lane * per; k < per && i < n; ++k, ++i) {
    const float m = mass[i];
    const float nc = __fadd_rn(cum, m);
    if (m > 0.f) {
      if (hit < 0 && nc > target) {
        hit = i;
        hb = cum;
      }
      lpos = i;
      lb = cum;
    }
    cum = nc;
  }
  int idx = -1;
  float before = 0.f;
  bool f = false;
  const uint32_t mh = __ballot_sync(0xffffffffu, hit >= 0);
  if (mh) {
    const int src = __ffs(mh) - 1;
    idx = __shfl_sync(0xffffffffu, hit, src);
    before = __shfl_sync(0xffffffffu, hb, src);
  } else {
    const uint32_t ml = __ballot_sync(0xffffffffu, lpos >= 0);
    if (ml) {
      const int src = 31 - __clz(ml);
      idx = __shfl_sync(0xffffffffu, lpos, src);
      before = __shfl_sync(0xffffffffu, lb, src);
      f = true;
    }
  }
  *rem = __fsub_rn(target, before);
  *Wout = W;
  *fb = f;
  return (W > 0.f) ? idx : -1;
}

// Membership of element (z, idx) in the top-F set whose smallest key is keyF.
SSD_DEV bool in_set(float z, int idx, float vF, uint64_t keyF) {
  return !(z < vF) && cand_key(z, idx) >= keyF;
}
SSD_DEV float norm_N(float C, float sq) { return __fsub_rn(1.f, __fmul_rn(__fsub_rn(1.f, C), sq)); }

// Element weights of the draws.  operator()(zt, zd, idx, Mk) -> weight >= 0,
// with Mk = fl(segment max kT) for the weights of the statistics pass; the
// passes and the draws compute them with the same operations.
struct WDraft {  // unnormalised q'_i relative to the segment maximum
  float kT, C, vF;
  uint64_t keyF;
  bool S;
  SSD_DEV float operator()(float, float zd, int idx, float Mk) const {
    const float e = ex2(__fmaf_rn(zd, kT, -Mk));
    return (S && in_set(zd, idx, vF, keyF)) ? __fmul_rn(e, C) : e;
  }
};
struct WTarget {  // unnormalised p_i relative to the segment maximum
  float kT;
  SSD_DEV float operator()(float zt, float, int, float Mk) const { return ex2(__fmaf_rn(zt, kT, -Mk)); }
};
struct WResid {  // max(0, p_i - q'_i), both normalised
  float kT, Mtk, inv_st, Mdk, f1, fC, vF;
  uint64_t keyF;
  bool S;
  SSD_DEV float p(float zt) const { return __fmul_rn(ex2(__fmaf_rn(zt, kT, -Mtk)), inv_st); }
  SSD_DEV float q(float zd, int idx) const {
    return __fmul_rn(ex2(__fmaf_rn(zd, kT, -Mdk)), (S && in_set(zd, idx, vF, keyF)) ? fC : f1);
  }
  SSD_DEV float operator()(float zt, float zd, int idx, float) const {
    const float r = __fsub_rn(p(zt), q(zd, idx));
    return r > 0.f ? r : 0.f;
  }
};
struct WProb {  // p_i normalised (the fallback of a residual without mass)
  float kT, Mtk, inv_st;
  SSD_DEV float operator()(float zt, float, int, float) const { return __fmul_rn(ex2(__fmaf_rn(zt, kT, -Mtk)), inv_st); }
};
// The residual weights of a position from its record.
SSD_DEV WResid resid_weights(const VocabArgs &a, const PairRec &r, int F) {
  WResid w;
  w.kT = a.kT;
  w.Mtk = __fmul_rn(r.gm[kTgt], a.kT);
  w.inv_st = __frcp_rn(r.gs[kTgt]);
  w.Mdk = __fmul_rn(r.gm[kDft], a.kT);
  const float sN = __fmul_rn(r.gs[kDft], r.N);
  w.f1 = __frcp_rn(sN);
  w.fC = __fdiv_rn(a.C, sN);
  // at C = 1 both weights are the correctly rounded 1 / sN: the membership
  // test would not change a weight, so it is skipped
  w.S = F > 0 && a.C < 1.f;
  w.keyF = r.keyF;
  w.vF = cand_val(r.keyF);
  return w;
}

// One warp: the element of block g (vectors 32 g .. 32 g + 31) of the rows
// whose running weight (lane sums by lane_sum, lanes by a scan) first exceeds
// `target` with positive weight; when rounding leaves the target in a lane
// without such an element, that lane's last positive element; when no lane
// holds it, the block's last positive element.  *dist: the target's distance
// from the nearer edge of the chosen element's bin (0 for the fallbacks).
template <class E, class WF>
SSD_DEV int warp_find(const VocabArgs &a, const char *rowT, const char *rowD, int g, float target, const WF &wf,
                      float Mk, float *dist, float *zt_out = nullptr, float *zd_out = nullptr) {
  const int lane = threadIdx.x & 31;
  const int v = g * 32 + lane;
  float zt[E::kVec], zd[E::kVec], x[E::kVec];
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) zt[e] = zd[e] = 0.f;
  if (rowT) E::unpack(row_vec<E>(a, rowT, v), zt);
  if (rowD) E::unpack(row_vec<E>(a, rowD, v), zd);
  const int i0 = v * E::kVec;
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) x[e] = (i0 + e < a.V) ? wf(zt[e], zd[e], i0 + e, Mk) : 0.f;
  const float L = lane_sum<E::kVec>(x);
  const float incl = warp_incl_scan(L);
  float ex = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) ex = 0.f;
  float run = 0.f, edge = 0.f;
  int hit = -1, lpos = -1;
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) {
    const float before = __fadd_rn(ex, run);
    run = __fadd_rn(run, x[e]);
    if (x[e] > 0.f) {
      lpos = i0 + e;
      const float after = __fadd_rn(ex, run);
      if (hit < 0 && after > target) {
        hit = lpos;
        edge = fminf(__fsub_rn(target, before), __fsub_rn(after, target));
      }
    }
  }
  const bool cross = L > 0.f && __fadd_rn(ex, L) > target;
  const uint32_t mc = __ballot_sync(0xffffffffu, cross);
  int d;
  if (mc) {
    const int src = __ffs(mc) - 1;
    *dist = __shfl_sync(0xffffffffu, hit >= 0 ? fmaxf(edge, 0.f) : 0.f, src);
    d = __shfl_sync(0xffffffffu, hit >= 0 ? hit : lpos, src);
  } else {
    *dist = 0.f;
    d = lpos;
#pragma unroll
    for (int o = 16; o; o >>= 1) d = max(d, __shfl_xor_sync(0xffffffffu, d, o));
  }
  if (zt_out || zd_out) {  // the element's two values, from the lane that read it
    const int owner = (d >= 0) ? d / E::kVec - g * 32 : 0;
    float vt = 0.f, vd = 0.f;
#pragma unroll
    for (int e = 0; e < E::kVec; ++e)
      if (lane == owner && i0 + e == d) {
        vt = zt[e];
        vd = zd[e];
      }
    vt = __shfl_sync(0xffffffffu, vt, owner & 31);
    vd = __shfl_sync(0xffffffffu, vd, owner & 31);
    if (zt_out) *zt_out = vt;
    if (zd_out) *zd_out = vd;
  }
  return d;
}

// ===========================================================================
// k_stats: one warp per segment of a row
// ===========================================================================
// One warp: the statistics of segment sg of a row, specialised by what the
// row kind records (KK block maximum keys, KB block sums, KA the argmax):
// each kind runs code without the other kinds' paths.
template <class E, bool KK, bool KB, bool KA>
SSD_DEV void stats_segment(const VocabArgs &a, const RowSlot &rs, int sg, int slot, int b) {
  const int lane = threadIdx.x & 31;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const char *row = row_ptr(a, rs.tensor, b, rs.row, E::kSize);
  const int v0 = sg * kSegVec;
  // every load of the segment in flight at once
  uint4 w[kSegBlocks];
  if (v0 + kSegVec <= a.nfull) {  // warp-uniform: every vector of the segment is whole
    const char *p = row + static_cast<int64_t>(v0 + lane) * 16;
#pragma unroll
    for (int k = 0; k < kSegBlocks; ++k) w[k] = ld_stream(p + 512 * k);
  } else {
#pragma unroll
    for (int k = 0; k < kSegBlocks; ++k) {
      const int v = v0 + 32 * k + lane;
      w[k] = (v < a.nfull) ? ld_stream(row + static_cast<int64_t>(v) * 16) : neg_inf_vec<E>();
    }
  }
  if (a.nvec > a.nfull && a.nfull >= v0 && a.nfull < v0 + kSegVec && lane == ((a.nfull - v0) & 31)) {
    const int kk = (a.nfull - v0) >> 5;  // the row's partial last vector
    const uint4 t = row_vec<E>(a, row, a.nfull);
#pragma unroll
    for (int k = 0; k < kSegBlocks; ++k)
      if (k == kk) w[k] = t;
  }
  // pass 1: maxima (bf16: packed), block maximum keys (lane k < 8 keeps
  // block k's), the argmax's vector
  uint32_t bk = 0u;
  float m1 = NEG_INF;
  int k1 = -1;
  if constexpr (E::kSize == 2) {
    // a segment wholly inside the row needs no validity checks (warp-uniform)
    const bool full = v0 + kSegVec <= a.nvec;
    uint32_t mm = 0xFF80FF80u;
#pragma unroll
    for (int k = 0; k < kSegBlocks; ++k) {
      const uint32_t t = bmax2(bmax2(w[k].x, w[k].y), bmax2(w[k].z, w[k].w));
      mm = bmax2(mm, t);
      if (KK) {
        // the vector maximum's key from its bf16 bits: with the maximum in
        // both halves, negative values flipped and the others' sign bit set
        // give the upper half of the order-preserving key of its float value
        // (the lower half follows the upper one and is masked off when stored)
        const uint32_t m2 = bmax2(t, __byte_perm(t, 0, 0x1032));
        uint32_t key = m2 ^ (static_cast<uint32_t>(static_cast<int32_t>(m2) >> 31) | 0x80000000u);
        if (!full && v0 + 32 * k + lane >= a.nvec) key = 0u;
        key = __reduce_max_sync(0xffffffffu, key);
        if (lane == k) bk = key;
      }
      if (KA) {
        const float vm = fmaxf(__uint_as_float(t << 16), __uint_as_float(t & 0xFFFF0000u));
        const bool valid = full || v0 + 32 * k + lane < a.nvec;
        if (valid && (vm > m1 || k1 < 0)) {  // strictly larger: the first vector among equal maxima
          m1 = fmaxf(m1, vm);
          k1 = k;
        }
      }
    }
    if (!KA) m1 = fmaxf(__uint_as_float(mm << 16), __uint_as_float(mm & 0xFFFF0000u));
  } else {
#pragma unroll
    for (int k = 0; k < kSegBlocks; ++k) {
      const float vm = vec_max<E>(w[k]);
      const bool valid = v0 + 32 * k + lane < a.nvec;
      if (KK) {
        const uint32_t key = __reduce_max_sync(0xffffffffu, valid ? f2ord(vm) : 0u);
        if (lane == k) bk = key;
      }
      if (valid && (vm > m1 || k1 < 0)) {
        m1 = fmaxf(m1, vm);
        k1 = k;
      }
    }
  }
  const float wm = ord2f(__reduce_max_sync(0xffffffffu, f2ord(m1)));
  int wa = v0 * E::kVec;  // the segment's first index unless the argmax is tracked
  if (KA) {
    int idx = kNone;
    if (k1 >= 0 && m1 == wm) {
      uint4 wk = w[0];
#pragma unroll
      for (int k = 1; k < kSegBlocks; ++k)
        if (k == k1) wk = w[k];
      float f[E::kVec];
      E::unpack(wk, f);
#pragma unroll
      for (int e = E::kVec - 1; e >= 0; --e)
        if (f[e] == wm) idx = (v0 + 32 * k1 + lane) * E::kVec + e;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
    wa = (idx == kNone) ? v0 * E::kVec : idx;
  }
  // pass 2: sums of 2^(z kT - fl(wm kT)), two elements per packed FMA / ADD;
  // per block the lane's part in the association of lane_sum
  float ws = 0.f, bsv = 0.f, wt = 0.f;
  if (!a.greedy && wm != NEG_INF) {
    const float Mk = __fmul_rn(wm, a.kT);
    const uint64_t k2 = pack2(a.kT, a.kT), m2 = pack2(-Mk, -Mk);
    uint64_t acc = pack2(0.f, 0.f);
    float pr[kSegBlocks];
#pragma unroll
    for (int k = 0; k < kSegBlocks; ++k) {
      uint64_t accj = 0;
#pragma unroll
      for (int h = 0; h < E::kPairs; ++h) {
        float x0, x1;
        unpack2(fma2(E::pair(w[k], h), k2, m2), x0, x1);
        const uint64_t e2 = pack2(ex2(x0), ex2(x1));
        accj = (h == 0) ? e2 : add2(accj, e2);
      }
      acc = add2(acc, accj);
      float lo, hi;
      unpack2(accj, lo, hi);
      pr[k] = __fadd_rn(lo, hi);
    }
    if (KB) {
      bsv = warp_block_sums(pr);
      // lane k < 8 takes block k's sum; their total by a scan (warp_runs over 8 masses)
      const float bk8 = __shfl_sync(0xffffffffu, bsv, (lane & 7) * 4);
      wt = __shfl_sync(0xffffffffu, warp_incl_scan(lane < kSegBlocks ? bk8 : 0.f), 31);
    }
    float lo, hi;
    unpack2(acc, lo, hi);
    ws = warp_sum(__fadd_rn(lo, hi));
  }
  const size_t si = slot_index(a, b, slot);
  if (lane == 0)
    reinterpret_cast<int4 *>(a.seg)[si * a.nseg + sg] =
        make_int4(__float_as_int(wm), __float_as_int(ws), wa, __float_as_int(wt));
  if (KK && lane < kSegBlocks) a.bkey[si * a.nblk + sg * kSegBlocks + lane] = E::kSize == 2 ? bk & 0xFFFF0000u : bk;
  if (KB && (lane & 3) == 0) a.bsum[si * a.nblk + sg * kSegBlocks + (lane >> 2)] = bsv;
}

template <class E>
__global__ void __launch_bounds__(kStatWarps * 32, 8) k_stats(const __grid_constant__ VocabArgs a) {
  // k_pair may start launching once every CTA of this grid has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the start mark only: at 64 registers an end mark makes the statistics pass spill
  if (a.trace && threadIdx.x == 0)
    trace_start(a, (static_cast<long>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x,
                a.b0 + static_cast<int>(blockIdx.z), static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x));
  if (a.ready && a.hits && a.do_lookup && a.b0 == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
      threadIdx.x == 0)
    *a.hits = 0u;
  const int warp = threadIdx.x >> 5;
  const int sg = static_cast<int>(blockIdx.x) * kStatWarps + warp;
  const int slot = static_cast<int>(blockIdx.y);
  const int b = a.b0 + static_cast<int>(blockIdx.z);
  const RowSlot rs = a.slot[slot];
  if (sg >= a.nseg) return;
  switch ((rs.keys ? 1 : 0) | (rs.blocks ? 2 : 0) | (rs.arg ? 4 : 0)) {  // uniform per CTA
    case 0: stats_segment<E, false, false, false>(a, rs, sg, slot, b); break;
    case 1: stats_segment<E, true, false, false>(a, rs, sg, slot, b); break;
    case 2: stats_segment<E, false, true, false>(a, rs, sg, slot, b); break;
    case 3: stats_segment<E, true, true, false>(a, rs, sg, slot, b); break;
    case 4: stats_segment<E, false, false, true>(a, rs, sg, slot, b); break;
    case 5: stats_segment<E, true, false, true>(a, rs, sg, slot, b); break;
    case 6: stats_segment<E, false, true, true>(a, rs, sg, slot, b); break;
    default: stats_segment<E, true, true, true>(a, rs, sg, slot, b); break;
  }
}

// ===========================================================================
// k_pair: one CTA per row pair
// ===========================================================================
struct __align__(16) PairSh {
  float gm[2], gs[2];  // row maximum and sum of 2^(z kT - fl(gm kT))
  int ga[2];           // row argmax
  float sq;            // the draft's normalised mass on S
  int ncand, nblist;
  alignas(16) uint32_t hist[2][256];
  uint64_t S[kMaxF];
  uint64_t cand[kCandCap];
  int blist[2 * kCandCap];
  uint64_t redk[kWarps];
  unsigned long long mk[8];
};
// Dynamic shared memory after PairSh: the target and draft rows' segment
// records, the draft's block keys, the drawn row's block masses and its
// segment masses.
struct PairBufs {
  SegRec *segT, *segD;
  uint32_t *keys;
  float *bm;   // block masses of the drawn row (segment units)
  float *smm;  // segment masses (row units); scratch of the row merges
};
__host__ __device__ inline size_t pair_smem_bytes(int nseg, int nblk) {
  return sizeof(PairSh) + 2 * static_cast<size_t>(nseg) * sizeof(SegRec) + 2 * static_cast<size_t>(nblk) * 4 +
         static_cast<size_t>(nseg) * 4;
}
SSD_DEV PairBufs pair_bufs(const VocabArgs &a, uint8_t *base) {
  PairBufs p;
  uint8_t *o = base;
  p.segT = reinterpret_cast<SegRec *>(o);
  o += static_cast<size_t>(a.nseg) * sizeof(SegRec);
  p.segD = reinterpret_cast<SegRec *>(o);
  o += static_cast<size_t>(a.nseg) * sizeof(SegRec);
  p.keys = reinterpret_cast<uint32_t *>(o);
  o += static_cast<size_t>(a.nblk) * sizeof(uint32_t);
  p.bm = reinterpret_cast<float *>(o);
  o += static_cast<size_t>(a.nblk) * sizeof(float);
  p.smm = reinterpret_cast<float *>(o);
  return p;
}

// One warp over a row's segment records (every lane returns the results):
// the maximum, the lowest index holding it, and the sum in units of
// fl(max kT) (each lane its segments in order, then a butterfly).
SSD_DEV void merge_row(const VocabArgs &a, const SegRec *sr, float &M, float &S, int &A) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int lane = threadIdx.x & 31;
  float m = NEG_INF;
  int am = kNone;
  for (int s = lane; s < a.nseg; s += 32) {
    const float ms = sr[s].m;
    if (ms > m) {  // a lane's segments in order: a strictly larger maximum keeps the lowest index
      m = ms;
      am = sr[s].a;
    }
  }
  M = ord2f(__reduce_max_sync(0xffffffffu, f2ord(m)));
  const unsigned ai = __reduce_min_sync(0xffffffffu, (m == M) ? static_cast<unsigned>(am) : static_cast<unsigned>(kNone));
  A = (ai == static_cast<unsigned>(kNone)) ? 0 : static_cast<int>(ai);
  float sum = 0.f;
  if (!a.greedy && M != NEG_INF) {
    const float Mk = __fmul_rn(M, a.kT);
    for (int s = lane; s < a.nseg; s += 32) {
      const SegRec r = sr[s];
      if (r.m != NEG_INF) sum = __fadd_rn(sum, __fmul_rn(r.s, ex2(__fsub_rn(__fmul_rn(r.m, a.kT), Mk))));
    }
    sum = warp_sum(sum);
  }
  S = sum;
}

// The elements (key prefix >= t16) of candidate block g of a draft row.
template <class E>
SSD_DEV void block_candidates(const VocabArgs &a, const char *row, int g, uint32_t t16, PairSh &sh) {
  const int lane = threadIdx.x & 31;
  const int v = g * 32 + lane;
  if (v >= a.nvec) return;
  float f[E::kVec];
  E::unpack(row_vec<E>(a, row, v), f);
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) {
    const int idx = v * E::kVec + e;
    if (idx < a.V && (f2ord(f[e]) >> 16) >= t16) {
      const int p = atomicAdd(&sh.ncand, 1);
      if (p < kCandCap) sh.cand[p] = cand_key(f[e], idx);
    }
  }
}

// The warps of k_pair that select the top-F list (warp 0 draws meanwhile):
// warps 1..7, synchronised by named barrier 1.
constexpr int kTopWarps = kWarps - 1;
constexpr int kTopThreads = kTopWarps * 32;
SSD_DEV void top_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kTopThreads) : "memory"); }

// Top-F of n distinct nonzero keys by rank (the key with r larger keys goes
// to dst[r] when r < F); slots past n are set to 0.  The top-F warps; no
// barrier inside.
SSD_DEV void rank_select(const uint64_t *keys, int n, int F, uint64_t *dst) {
  const int gt = threadIdx.x - 32, gw = gt >> 5, lane = threadIdx.x & 31;
  for (int i = gt; i < F; i += kTopThreads)
    if (i >= n) dst[i] = 0ull;
  if (n <= 64) {
    const uint64_t a0 = lane < n ? keys[lane] : 0ull, a1 = lane + 32 < n ? keys[lane + 32] : 0ull;
    for (int i = gw; i < n; i += kTopWarps) {
      const uint64_t k = keys[i];
      const int rank = __popc(__ballot_sync(0xffffffffu, a0 > k)) + __popc(__ballot_sync(0xffffffffu, a1 > k));
      if (lane == 0 && rank < F) dst[rank] = k;
    }
    return;
  }
  for (int i = gt; i < n; i += kTopThreads) {
    const uint64_t k = keys[i];
    int rank = 0;
    for (int j = 0; j < n && rank < F; ++j) rank += (keys[j] > k) ? 1 : 0;
    if (rank < F) dst[rank] = k;
  }
}

// One warp (every lane returns the result): over 256 bucket counts, the
// bucket where the count from the top bucket down first reaches `need` and
// the count in the buckets above it; when the total stays below `need`,
// bucket 0 and the count above bucket 0.  Lane l holds buckets 255 - 8l down
// to 248 - 8l.
SSD_DEV void find_bucket(const uint32_t *hist, int need, uint32_t &bucket_out, int &above_out) {
  const int lane = threadIdx.x & 31;
  const int hi = 255 - 8 * lane;
  const uint4 x = *reinterpret_cast<const uint4 *>(hist + hi - 7);
  const uint4 y = *reinterpret_cast<const uint4 *>(hist + hi - 3);
  const uint32_t c[8] = {y.w, y.z, y.y, y.x, x.w, x.z, x.y, x.x};  // buckets hi, hi - 1, ..., hi - 7
  uint32_t tot = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) tot += c[k];
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const uint32_t n = static_cast<uint32_t>(need);
  const uint32_t m = __ballot_sync(0xffffffffu, incl >= n);
  int bucket = 0;
  uint32_t above = 0;
  if (m) {
    const int src = __ffs(m) - 1;
    if (lane == src) {
      uint32_t run = incl - tot;
      int k = 7;
      bool found = false;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (!found && (q == 7 || run + c[q] >= n)) {
          k = q;
          found = true;
        } else if (!found) {
          run += c[q];
        }
      }
      bucket = hi - k;
      above = run;
    }
    bucket = __shfl_sync(0xffffffffu, bucket, src);
    above = __shfl_sync(0xffffffffu, above, src);
  } else {
    above = __shfl_sync(0xffffffffu, incl, 31) - __shfl_sync(0xffffffffu, c[7], 31);
  }
  bucket_out = static_cast<uint32_t>(bucket);
  above_out = static_cast<int>(above);
}

// The top-F (F > 1) of a draft row into sh.S (descending; zeros past the
// row's elements), by the top-F warps.  t16 = the 16-bit key prefix of the
// F-th largest block maximum (two levels of 256-bucket counts): at least F
// elements reach it, so the row's top-F all lie in blocks whose maximum does.
// Those blocks are read again (one warp per block) and their elements
// reaching t16 ranked; when ties overflow the buffers, F sweeps of a group
// maximum instead.
template <class E>
SSD_DEV void row_topf(const VocabArgs &a, const char *row, int F, const uint32_t *keys, PairSh &sh) {
  const int gt = threadIdx.x - 32, gw = gt >> 5, lane = threadIdx.x & 31;
  const int nb = a.nblk;
  auto count = [&](uint32_t *hist, bool v, uint32_t bucket) {
    const uint32_t peers = __match_any_sync(0xffffffffu, v ? bucket : 0xFFFFFFFFu);
    if (v && lane == __ffs(peers) - 1) atomicAdd(&hist[bucket], static_cast<uint32_t>(__popc(peers)));
  };
  for (int i = gt; i < 512; i += kTopThreads) sh.hist[i >> 8][i & 255] = 0u;
  if (gt == 0) {
    sh.ncand = 0;
    sh.nblist = 0;
  }
  top_sync();
  for (int i0 = gw * 32; i0 < nb; i0 += kTopThreads) {
    const uint32_t k = (i0 + lane < nb) ? keys[i0 + lane] : 0u;
    count(sh.hist[0], k != 0u, k >> 24);
  }
  top_sync();
  uint32_t b1, b2;
  int above, above2;
  find_bucket(sh.hist[0], F, b1, above);
  for (int i0 = gw * 32; i0 < nb; i0 += kTopThreads) {
    const uint32_t k = (i0 + lane < nb) ? keys[i0 + lane] : 0u;
    count(sh.hist[1], k != 0u && (k >> 24) == b1, (k >> 16) & 0xFFu);
  }
  top_sync();
  find_bucket(sh.hist[1], F - above, b2, above2);
  const uint32_t t16 = (b1 << 8) | b2;
  constexpr int kListCap = 2 * kCandCap;
  for (int i = gt; i < nb; i += kTopThreads) {
    const uint32_t k = keys[i];
    if (k && (k >> 16) >= t16) {
      const int p = atomicAdd(&sh.nblist, 1);
      if (p < kListCap) sh.blist[p] = i;
    }
  }
  top_sync();
  const int nbl = sh.nblist;
  const bool listed = nbl <= kListCap;
  if (listed)
    for (int q = gw; q < nbl; q += kTopWarps) block_candidates<E>(a, row, sh.blist[q], t16, sh);
  top_sync();
  const int nc = sh.ncand;
  if (listed && nc <= kCandCap) {
    rank_select(sh.cand, nc, F, sh.S);
  } else {
    // ties at the threshold: one winner per sweep over the candidate blocks
    // (every block when they overflow the list)
    const int nq = listed ? nbl : nb;
    uint64_t prev = ~0ull;
    for (int r = 0; r < F; ++r) {
      uint64_t best = 0ull;
      for (int q = gw; q < nq; q += kTopWarps) {
        const int g = listed ? sh.blist[q] : q;
        const int v = g * 32 + lane;
        if (v >= a.nvec) continue;
        float f[E::kVec];
        E::unpack(row_vec<E>(a, row, v), f);
#pragma unroll
        for (int e = 0; e < E::kVec; ++e) {
          const int idx = v * E::kVec + e;
          if (idx >= a.V || (f2ord(f[e]) >> 16) < t16) continue;
          const uint64_t key = cand_key(f[e], idx);
          if (key < prev && key > best) best = key;
        }
      }
      best = warp_max_u64(best);
      if (lane == 0) sh.redk[gw] = best;
      top_sync();
      best = sh.redk[0];
      for (int w = 1; w < kTopWarps; ++w) best = sh.redk[w] > best ? sh.redk[w] : best;
      top_sync();
      if (gt == 0) sh.S[r] = best;
      prev = best;
    }
  }
  top_sync();
}

// One warp: inverse-CDF draw over a row from its segment masses smm (row
// units), block masses bm (segment units: weights relative to fl(seg max kT))
// and a warp_find over the located block, which reads both rows' vectors
// when given.  Returns the element (every lane; -1 when the row has no
// weight) with its target / draft values and whether it is a near-tie.
template <class E, class WF>
SSD_DEV int row_draw(const VocabArgs &a, const SegRec *sr, float rowMk, const float *smm, const float *bm,
                     const char *rowT, const char *rowD, float u, const WF &wf, bool *near, float *zt, float *zd) {
  float rem, W;
  bool fb;
  const int s = warp_locate(smm, a.nseg, u, false, &rem, &W, &fb);
  *near = true;
  if (s < 0) return -1;
  const float Ms = __fmul_rn(sr[s].m, a.kT);
  const float f = ex2(__fsub_rn(Ms, rowMk));  // a segment unit in row units
  float rem2, W2;
  bool fb2;
  const int k = warp_locate(bm + s * kSegBlocks, kSegBlocks, __fdiv_rn(rem, f), true, &rem2, &W2, &fb2);
  if (k < 0) return -1;
  float dist;
  const int d = warp_find<E>(a, rowT, rowD, s * kSegBlocks + k, rem2, wf, Ms, &dist, zt, zd);
  *near = fb || fb2 || d < 0 || !(__fmul_rn(dist, f) >= __fmul_rn(kNearTie, W));
  return d;
}

// CS: C < 1 (the draft's draws weighted by the top-F set); at C = 1 the kernel
// has no code for the weighted draw.
template <class E, bool CS>
__global__ void __launch_bounds__(kThreads) k_pair(const __grid_constant__ VocabArgs a) {
  // k_resid (if any) may start launching once every CTA of this grid has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(16) uint8_t pair_smem[];
  PairSh &sh = *reinterpret_cast<PairSh *>(pair_smem);
  const PairBufs pb = pair_bufs(a, pair_smem + sizeof(PairSh));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = static_cast<int>(blockIdx.x) / a.npairs;
  const int j = static_cast<int>(blockIdx.x) - b * a.npairs;
  const int K = a.K;
  const float NEG_INF = -__int_as_float(0x7f800000);
  if (a.trace && tid == 0) {
    for (int k = 0; k < 8; ++k) sh.mk[k] = 0ull;
    sh.mk[1] = now_ns();
  }
  const int ts = a.tsl[j], ds = a.dsl[j];
  const bool hT = ts >= 0, hD = ds >= 0;
  const int F = hD ? a.Fs[j] : 0;
  const bool greedy = a.greedy != 0;
  const bool sampled = a.do_sample && j < K;
  const bool tested = a.do_verify && j < K;
  const bool bonus_p = a.do_verify && j == K && !greedy;
  // C < 1 weights the draft's draw by S: it waits for the top-F list
  const bool weighted = CS && !greedy && sampled && F > 0;
  // with C = 1 (or greedy) the record does not depend on S (N = 1, and in or
  // out of S the draft's weight is the same): it is published before the top-F
  const bool early = a.ready != nullptr && (greedy || !CS);
  const char *rowT = row_ptr(a, 0, b, j, E::kSize);
  const char *rowD = row_ptr(a, 1, b, j, E::kSize);
  // the counters k_resid takes tickets on and the hit count start at zero
  // (k_resid waits for this grid to complete before it touches them)
  if (tid == 0) {
    if (j == 0) a.ctr[2 + b] = 0u;
    if (j < K && a.do_analytics) a.ctr[2 + a.B + static_cast<size_t>(b) * K + j] = 0u;
    if (!a.ready && b == 0 && j == 0 && a.do_lookup && a.hits) *a.hits = 0u;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");  // k_stats has completed
  if (a.trace && tid == 0) sh.mk[2] = now_ns();
  // stage the records
  const int drawn = (sampled && !greedy) ? kDft : (bonus_p ? kTgt : -1);
  {
    const int4 *sT = reinterpret_cast<const int4 *>(a.seg + slot_index(a, b, hT ? ts : 0) * a.nseg);
    const int4 *sD = reinterpret_cast<const int4 *>(a.seg + slot_index(a, b, hD ? ds : 0) * a.nseg);
    for (int s = tid; s < a.nseg; s += kThreads) {
      if (hT) cp_async16(pb.segT + s, sT + s);
      if (hD) cp_async16(pb.segD + s, sD + s);
    }
    if (F >= 2) {
      const uint32_t *k = a.bkey + slot_index(a, b, ds) * a.nblk;
      for (int i = tid; i < a.nblk / 4; i += kThreads)
        cp_async16(reinterpret_cast<int4 *>(pb.keys) + i, reinterpret_cast<const int4 *>(k) + i);
    }
    if (drawn >= 0) {
      const float *bs = a.bsum + slot_index(a, b, drawn == kDft ? ds : ts) * a.nblk;
      for (int i = tid; i < a.nblk / 4; i += kThreads)
        cp_async16(reinterpret_cast<int4 *>(pb.bm) + i, reinterpret_cast<const int4 *>(bs) + i);
    }
    cp_async_wait_all();
  }
  if (tid == 0) {
    if (!hT) sh.gm[kTgt] = sh.gs[kTgt] = 0.f, sh.ga[kTgt] = 0;
    if (!hD) sh.gm[kDft] = sh.gs[kDft] = 0.f, sh.ga[kDft] = 0;
  }
  __syncthreads();
  if (a.trace && tid == 0) sh.mk[3] = now_ns();
  // row statistics: warp 0 the target row, warp 1 the draft row
  if ((warp == 0 && hT) || (warp == 1 && hD)) {
    float M, S;
    int A;
    merge_row(a, warp == 0 ? pb.segT : pb.segD, M, S, A);
    if (lane == 0) {
      sh.gm[warp] = M;
      sh.gs[warp] = S;
      sh.ga[warp] = A;
    }
  }
  __syncthreads();
  if (a.trace && tid == 0) sh.mk[4] = now_ns();
  const float mtk = __fmul_rn(sh.gm[kTgt], a.kT), mdk = __fmul_rn(sh.gm[kDft], a.kT);
  const int at = sh.ga[kTgt], ad = sh.ga[kDft];
  // the drawn row's segment masses in row units (from the segment totals)
  const SegRec *srd = drawn == kDft ? pb.segD : pb.segT;
  const float rowMk = drawn == kDft ? mdk : mtk;
  if (drawn >= 0 && !weighted) {
    for (int s = tid; s < a.nseg; s += kThreads) {
      const float m = srd[s].m;
      pb.smm[s] = (m == NEG_INF) ? 0.f : __fmul_rn(srd[s].t, ex2(__fsub_rn(__fmul_rn(m, a.kT), rowMk)));
    }
    __syncthreads();
  }
  // warp 0 keeps the position's record
  PairRec r;
  memset(&r, 0, sizeof(r));
  r.d = -1;
  r.bt = -1;
  r.W = 1.f;
  r.N = 1.f;
  // the draw of d_{j+1} (or the given token) with p(d) and q(d) when it does
  // not depend on S, and the bonus after full acceptance
  float zt = 0.f, zd = 0.f;
  bool zknown = false;
  if (warp == 0) {
    if (sampled || tested) {
      int d;
      bool near = false;
      if (sampled && greedy) {
        d = ad;
      } else if (sampled && !weighted) {
        const WDraft wd{a.kT, 1.f, 0.f, 0ull, false};
        d = row_draw<E>(a, pb.segD, mdk, pb.smm, pb.bm, hT ? rowT : nullptr, rowD,
                        a.u_draft[static_cast<size_t>(b) * K + j], wd, &near, &zt, &zd);
        zknown = d >= 0;
        if (d < 0) {
          d = ad;
          near = true;
        }
      } else if (sampled) {
        d = -1;  // drawn once S is known
      } else {
        d = a.d_in[static_cast<size_t>(b) * K + j];
      }
      r.d = d;
      if (near) r.fl |= kRecDrawNear;
    }
    if (a.do_verify && j == K) {
      if (greedy) {
        r.bt = at;
      } else {
        bool near;
        float z0, z1;
        int bt = row_draw<E>(a, pb.segT, mtk, pb.smm, pb.bm, rowT, nullptr, a.u_bonus[b], WTarget{a.kT}, &near, &z0,
                             &z1);
        if (bt < 0) {
          bt = at;
          near = true;
        }
        r.bt = bt;
        if (near) r.fl |= kRecBonusNear;
      }
    }
  }
  if (a.trace && tid == 0) sh.mk[5] = now_ns();
  // p(d), q'(d), the verdict, the outputs and the record (warp 0); with the
  // ready words the record is published (release) right after it is written
  auto finish = [&](float N, uint64_t keyF) {
    r.N = N;
    r.keyF = keyF;
    r.gm[kTgt] = sh.gm[kTgt];
    r.gm[kDft] = sh.gm[kDft];
    r.gs[kTgt] = sh.gs[kTgt];
    r.gs[kDft] = sh.gs[kDft];
    if (sampled || tested) {
      const int d = r.d;
      if (d >= 0 && d < a.V) {
        if (greedy) {
          r.p = (d == at) ? 1.f : 0.f;
          r.q = (d == ad) ? 1.f : 0.f;
        } else {
          if (!zknown) {
            zd = E::ld(rowD, d);
            zt = hT ? E::ld(rowT, d) : 0.f;
          }
          const bool ins = F > 0 && cand_key(zd, d) >= keyF;
          const float q = __fdiv_rn(ex2(__fmaf_rn(zd, a.kT, -mdk)), sh.gs[kDft]);
          r.q = __fdiv_rn(ins ? __fmul_rn(q, a.C) : q, N);
          if (hT) r.p = __fdiv_rn(ex2(__fmaf_rn(zt, a.kT, -mtk)), sh.gs[kTgt]);
        }
      } else {
        r.p = -1.f;
        r.q = 0.f;
        if (lane == 0) atomicOr(a.status, kFlagBadToken);
      }
      if (tested && r.p >= 0.f && __fmul_rn(a.u_acc[static_cast<size_t>(b) * K + j], r.q) < r.p)
        r.fl |= kRecAccepted;
      if (tested) r.bt = at;  // greedy: the bonus; T > 0: the residual draw's fallback
      if (tested && greedy) {
        r.W = (at != ad) ? 1.f : 0.f;
        if (!(r.W > 0.f)) r.fl |= kRecZero;
      }
    }
    if (lane == 0) {
      if (sampled) {
        a.d_out[static_cast<size_t>(b) * K + j] = r.d;
        if (a.qd_out) a.qd_out[static_cast<size_t>(b) * K + j] = r.q;
        if (a.fill_payload) a.fill_payload[static_cast<size_t>(b) * a.fill_stride + a.fill_col] = r.d;
      }
      if (tested && a.accept_prob) {
        float ap;
        if (r.p < 0.f) ap = 0.f;
        else if (r.q > 0.f) ap = fminf(1.f, __fdiv_rn(r.p, r.q));
        else ap = (r.p > 0.f) ? 1.f : 0.f;
        a.accept_prob[static_cast<size_t>(b) * K + j] = ap;
      }
      if (a.do_verify) a.rec[static_cast<size_t>(b) * (K + 1) + j] = r;
      if (a.ready) publish_ready(&a.ready[(static_cast<size_t>(b) * (K + 1) + j) * 2]);
      if (a.do_analytics) {
        // the hit partials come from warp 1 (below); the rest of the record here
        PairRec *dst = a.rec + static_cast<size_t>(b) * (K + 1) + j;
        dst->N = r.N;
        dst->keyF = r.keyF;
        dst->gm[0] = r.gm[0];
        dst->gm[1] = r.gm[1];
        dst->gs[0] = r.gs[0];
        dst->gs[1] = r.gs[1];
      }
    }
  };
  if (early && warp == 0) finish(1.f, 0ull);
  // the draft row's top-F list S (warps 1..7, while warp 0 draws), its
  // normalised mass and the guesses of depth j
  if (F == 1 && tid == 0) sh.S[0] = cand_key(sh.gm[kDft], ad);
  if (F >= 2 && warp > 0) row_topf<E>(a, rowD, F, pb.keys, sh);
  __syncthreads();
  if (warp == 1) {
    float sq = 0.f;
    if (!greedy && F > 0 && sh.gm[kDft] != NEG_INF) {
      for (int i = lane; i < F; i += 32)
        if (sh.S[i]) sq = __fadd_rn(sq, ex2(__fmaf_rn(cand_val(sh.S[i]), a.kT, -mdk)));
      sq = __fdiv_rn(warp_sum(sq), sh.gs[kDft]);
    }
    if (lane == 0) sh.sq = sq;
  }
  if (a.do_predict && hD) {
    const int sumF = a.foff[K + 1];
    for (int i = tid; i < a.F[j]; i += kThreads) {
      const uint64_t key = sh.S[i];
      a.guess[static_cast<size_t>(b) * sumF + a.foff[j] + i] = cand_idx(key);
      if (a.guess_q) {
        float q;
        if (greedy) q = (i == 0) ? 1.f : 0.f;
        else q = __fdiv_rn(ex2(__fmaf_rn(cand_val(key), a.kT, -mdk)), sh.gs[kDft]);
        a.guess_q[static_cast<size_t>(b) * sumF + a.foff[j] + i] = q;
      }
    }
  }
  __syncthreads();
  if (a.ready && tid == 0) {  // the guess list of depth j is written
    __threadfence();
    publish_ready(&a.ready[(static_cast<size_t>(b) * (K + 1) + j) * 2 + 1]);
  }
  if (a.trace && tid == 0) sh.mk[6] = now_ns();
  const uint64_t keyF = F > 0 ? sh.S[F - 1] : 0ull;
  const float vF = cand_val(keyF);
  const float N = norm_N(a.C, sh.sq);
  if (weighted) {
    // the Saguaro weights: block masses with the elements of S down-weighted
    // (in list order), segment masses in row units from them
    for (int i = tid; i < a.nblk; i += kThreads) {
      float m = pb.bm[i];
      const float Ms = __fmul_rn(srd[i / kSegBlocks].m, a.kT);
      for (int t = 0; t < F; ++t) {
        const uint64_t key = sh.S[t];
        if (!key || (cand_idx(key) / E::kVec) / 32 != i) continue;
        m = __fsub_rn(m, __fmul_rn(__fsub_rn(1.f, a.C), ex2(__fmaf_rn(cand_val(key), a.kT, -Ms))));
      }
      pb.bm[i] = fmaxf(m, 0.f);
    }
    __syncthreads();
    for (int s = warp; s < a.nseg; s += kWarps) {
      const float t = warp_total(pb.bm + s * kSegBlocks, kSegBlocks);
      if (lane == 0) {
        const float m = srd[s].m;
        pb.smm[s] = (m == NEG_INF) ? 0.f : __fmul_rn(t, ex2(__fsub_rn(__fmul_rn(m, a.kT), rowMk)));
      }
    }
    __syncthreads();
    if (warp == 0) {
      const WDraft wd{a.kT, a.C, vF, keyF, true};
      bool near;
      int d = row_draw<E>(a, pb.segD, mdk, pb.smm, pb.bm, hT ? rowT : nullptr, rowD,
                          a.u_draft[static_cast<size_t>(b) * K + j], wd, &near, &zt, &zd);
      zknown = d >= 0;
      if (d < 0) {
        d = ad;
        near = true;
      }
      r.d = d;
      if (near) r.fl |= kRecDrawNear;
    }
  }
  if (!early && warp == 0) finish(N, keyF);

  // analytics: the guesses' target and residual probability (all of S carries C in q')
  if (a.do_analytics && warp == 1) {
    float hp = 0.f, hr = 0.f;
    if (greedy) {
      for (int i = lane; i < a.F[j]; i += 32)
        if (cand_idx(sh.S[i]) == at) hp = 1.f;
      hp = warp_max(hp);
      hr = hp;
    } else {
      const float inv_st = __frcp_rn(sh.gs[kTgt]);
      const float fC = __fdiv_rn(a.C, __fmul_rn(sh.gs[kDft], N));
      for (int i = lane; i < a.F[j]; i += 32) {
        const uint64_t key = sh.S[i];
        if (!key) continue;
        const int d = cand_idx(key);
        const float p = __fmul_rn(ex2(__fmaf_rn(E::ld(rowT, d), a.kT, -mtk)), inv_st);
        hp = __fadd_rn(hp, p);
        if (j < K) {
          const float q = __fmul_rn(ex2(__fmaf_rn(cand_val(key), a.kT, -mdk)), fC);
          hr = __fadd_rn(hr, fmaxf(__fsub_rn(p, q), 0.f));
        }
      }
      hp = warp_sum(hp);
      hr = warp_sum(hr);
    }
    if (lane == 0) {
      PairRec *dst = a.rec + static_cast<size_t>(b) * (K + 1) + j;
      dst->hp = hp;
      dst->hr = hr;
      float al = 0.f, W = 0.f;
      if (greedy) {
        al = (j < K && at == ad) ? 1.f : 0.f;
        W = 1.f - al;
      }
      dst->al = al;
      dst->W = W;
    }
  }
  if (a.trace && tid == 0) {
    sh.mk[7] = now_ns();
    trace_entry(a, a.trace_pair + blockIdx.x, 1, b, j, sh.mk);
  }
}

// ===========================================================================
// k_resid: residual units, the bonus draw and the sequence finish
// ===========================================================================
constexpr int kLookupStage = 2048;  // guesses + payload words of a sequence staged in shared memory
struct __align__(16) ResSh {
  PairRec rec[kMaxK + 1];
  float u[kMaxK];
  float seg[kMaxSub * kWarps][2];  // this unit's half-segment masses (residual, p) per group, or its warps' analytics sums
  float um[2][kMaxUnits];    // the sequence's unit masses (residual, p)
  float bx[kUnitSeg * kSegBlocks];
  float sm[kMaxSub * kResSeg];   // the located unit's segment masses
  float scal[4];
  int ival[4];
  unsigned long long mk[8];
};
// The residual pass's vectors: per warp its half segment of both rows (4
// blocks of 32 vectors), staged by cp.async so that the block loop need not be
// unrolled.  Once the pass is done the finishing unit reuses the space for the
// final draw's blocks, the segment masses and the lookup lists, so that a unit
// CTA stays small and every unit of the grid is resident early.
struct __align__(16) ResStage {
  union {
    uint4 v[kWarps][2][kSegBlocks / 2][32];
    struct {
      uint4 blk[kWarps][2][32];      // the final draw: one block of both rows per warp
      float2 sgm[kMaxSeg];           // the sequence's segment masses (residual, p)
      int32_t look[kLookupStage];    // the sequence's guesses, then its payload
    } fin;
  };
};

// The outputs of sequence b once its bonus token bt is known (sh.rec: its
// records, sh.u: its acceptance uniforms, look: its lookup lists when
// `staged`).
SSD_DEV void emit(const VocabArgs &a, int b, int acc, int bt, float W, bool zero, bool near_bonus, bool staged,
                  ResSh &sh, const int32_t *look) {
  const int tid = threadIdx.x;
  const int K = a.K;
  const int sumF = a.foff[K + 1];
  if (tid == 0) {
    sh.ival[3] = kNone;
    if (a.near_ties && !a.greedy) {
      // the acceptance tests actually taken (positions 1..acc+1) whose u
      // lies within kNearTie of p/q', the bonus draw and (sampling) the
      // draws of d_1..d_K
      uint32_t n = near_bonus ? 1u : 0u;
      for (int t = 0; t <= acc && t < K; ++t) {
        const PairRec &r = sh.rec[t];
        if (r.p >= 0.f && r.q > 0.f && fabsf(__fsub_rn(sh.u[t], __fdiv_rn(r.p, r.q))) < kNearTie) ++n;
      }
      if (a.do_sample)
        for (int t = 0; t < K; ++t) n += (sh.rec[t].fl & kRecDrawNear) ? 1u : 0u;
      if (n) atomicAdd(a.near_ties, n);
    }
  }
  __syncthreads();
  if (a.do_lookup) {
    for (int i = tid; i < a.F[acc]; i += kThreads) {
      const int g = staged ? look[a.foff[acc] + i] : __ldcg(a.guess + static_cast<size_t>(b) * sumF + a.foff[acc] + i);
      if (g == bt) atomicMin(&sh.ival[3], i);
    }
    __syncthreads();
  }
  const int s_hit = (a.do_lookup && sh.ival[3] != kNone) ? a.foff[acc] + sh.ival[3] : -1;
  for (int t = tid; t <= K; t += kThreads) {
    int v = -1;
    if (t < acc) v = sh.rec[t].d;
    if (t == acc) v = bt;
    a.out_tokens[static_cast<size_t>(b) * (K + 1) + t] = v;
  }
  if (a.do_lookup && a.next_tokens)
    for (int t = tid; t < K; t += kThreads) {
      int v = -1;
      if (s_hit >= 0 && a.payload)
        v = staged ? look[sumF + s_hit * K + t] : a.payload[(static_cast<size_t>(b) * sumF + s_hit) * K + t];
      a.next_tokens[static_cast<size_t>(b) * K + t] = v;
    }
  if (tid == 0) {
    if (zero) atomicOr(a.status, kFlagZeroResidual);
    a.accept_len[b] = acc;
    a.bonus[b] = bt;
    if (a.resid_mass) a.resid_mass[b] = W;
    if (a.do_lookup) {
      if (a.slot_out) a.slot_out[b] = s_hit;
      if (s_hit >= 0 && a.hits) atomicAdd(a.hits, 1u);
    }
  }
}

// Stage nb blocks (32 vectors each) of row pair j of sequence b, from block
// g0 on, for warp `w` in st: all of the warp's loads in flight at once.
template <class E>
SSD_DEV void stage_blocks(const VocabArgs &a, int b, int j, int g0, int nb, int w, ResStage &st) {
  const int lane = threadIdx.x & 31;
  const char *rowT = row_ptr(a, 0, b, j, E::kSize);
  const char *rowD = row_ptr(a, 1, b, j, E::kSize);
  for (int k = 0; k < nb; ++k) {
    const int v = (g0 + k) * 32 + lane;
    if (v < a.nfull) {
      cp_async16(&st.v[w][0][k][lane], rowT + static_cast<int64_t>(v) * 16);
      cp_async16(&st.v[w][1][k][lane], rowD + static_cast<int64_t>(v) * 16);
    } else {
      st.v[w][0][k][lane] = row_vec<E>(a, rowT, v);
      st.v[w][1][k][lane] = row_vec<E>(a, rowD, v);
    }
  }
  cp_async_wait_all();
  __syncwarp();
}

// Stage block g of row pair j of sequence b for warp w into the final draw's
// space (every load the thread issued before, e.g. lookup lists, completes too).
template <class E>
SSD_DEV void stage_block1(const VocabArgs &a, int b, int j, int g, int w, ResStage &st) {
  const int lane = threadIdx.x & 31;
  const char *rowT = row_ptr(a, 0, b, j, E::kSize);
  const char *rowD = row_ptr(a, 1, b, j, E::kSize);
  const int v = g * 32 + lane;
  if (v < a.nfull) {
    cp_async16(&st.fin.blk[w][0][lane], rowT + static_cast<int64_t>(v) * 16);
    cp_async16(&st.fin.blk[w][1][lane], rowD + static_cast<int64_t>(v) * 16);
  } else {
    st.fin.blk[w][0][lane] = row_vec<E>(a, rowT, v);
    st.fin.blk[w][1][lane] = row_vec<E>(a, rowD, v);
  }
  cp_async_wait_all();
  __syncwarp();
}

// Residual pass over unit u of row pair j of sequence b: a.unit_sub groups of
// kResSeg segments (the unit's segments (u unit_sub + g) kResSeg .. + 3 in
// group g), two warps per segment, four blocks each.  Each lane sums max(0, p -
// q') and p over its elements in order, the lanes by a butterfly: the
// half-segment masses of group g into sh.seg[g kWarps + warp].  kMins: *mn,
// *mx (every lane) = the warp's sums of min(p, q') and of max(0, p - q') over
// the unit.  kS: the call has C < 1, so the draft's weights may test membership
// in the top-F set (at C = 1 the unit pass has no code for it).
template <class E, bool kMins, bool kS>
SSD_DEV void unit_pass(const VocabArgs &a, int b, int j, int u, const WResid &wr, ResSh &sh, ResStage &st,
                       float *mn_out, float *mx_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float mn = 0.f, mx = 0.f;
#pragma unroll 1
  for (int grp = 0; grp < a.unit_sub; ++grp) {
    const int sg = (u * a.unit_sub + grp) * kResSeg + (warp >> 1);
    const int g0 = sg * kSegBlocks + (warp & 1) * (kSegBlocks / 2);
    float rs = 0.f, ps = 0.f;
    if (sg < a.nseg) {
      stage_blocks<E>(a, b, j, g0, kSegBlocks / 2, warp, st);
#pragma unroll 1
      for (int k = 0; k < kSegBlocks / 2; ++k) {
        const int i0 = ((g0 + k) * 32 + lane) * E::kVec;
        float ft[E::kVec], fd[E::kVec];
        E::unpack(st.v[warp][0][k][lane], ft);
        E::unpack(st.v[warp][1][k][lane], fd);
#pragma unroll
        for (int e = 0; e < E::kVec; ++e) {
          if (i0 + e < a.V) {
            // wr.p and wr.q as one packed pair: per lane the same roundings
            float xt, xd, p, q;
            unpack2(fma2(pack2(ft[e], fd[e]), pack2(wr.kT, wr.kT), pack2(-wr.Mtk, -wr.Mdk)), xt, xd);
            const float fq = (kS && wr.S && in_set(fd[e], i0 + e, wr.vF, wr.keyF)) ? wr.fC : wr.f1;
            unpack2(mul2(pack2(ex2(xt), ex2(xd)), pack2(wr.inv_st, fq)), p, q);
            const float r = __fsub_rn(p, q);
            unpack2(add2(pack2(rs, ps), pack2(r > 0.f ? r : 0.f, p)), rs, ps);
            if (kMins) mn = __fadd_rn(mn, fminf(p, q));
          }
        }
      }
      rs = warp_sum(rs);
      ps = warp_sum(ps);
    }
    if (lane == 0) {
      sh.seg[grp * kWarps + warp][0] = rs;
      sh.seg[grp * kWarps + warp][1] = ps;
    }
    if (kMins) mx = __fadd_rn(mx, rs);
  }
  if (kMins) {
    *mn_out = warp_sum(mn);
    *mx_out = mx;
  }
}

// The last residual unit of sequence b, every thread: the bonus from max(0,
// p - q') of pair acc (p when the residual has no mass).  Warp 0 locates the
// unit (sh.um) and the segment (st.fin.sgm); the eight warps read the segment's
// blocks again, one each, for their sums (lane sums, then a scan: the
// arithmetic of the element search); warp 0 locates the block and the
// element.  Returns the token (-1: no weight); sets *W (the residual mass),
// *zero and *near.
template <class E>
SSD_DEV int resid_draw(const VocabArgs &a, int b, int acc, const WResid &wr, ResSh &sh, ResStage &st, float *W_out,
                       bool *zero, bool *near) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int U = a.nunits;
  if (warp == 0) {
    const float W0 = warp_total(sh.um[0], U);
    const int X = (W0 > 0.f) ? 0 : 1;
    float rem, W;
    bool fb;
    const int q = warp_locate(sh.um[X], U, a.u_bonus[b], false, &rem, &W, &fb);
    int sg = -1;
    float rem2 = 0.f, W2;
    bool fb2 = false;
    if (q >= 0) {
      const int nus = a.unit_sub * kResSeg;  // the unit's segments (<= 32)
      if (lane < nus) {
        const int t = q * nus + lane;
        sh.sm[lane] = (t < a.nseg) ? (X ? st.fin.sgm[t].y : st.fin.sgm[t].x) : 0.f;
      }
      __syncwarp();
      const int s = warp_locate(sh.sm, nus, rem, true, &rem2, &W2, &fb2);
      if (s >= 0) sg = q * nus + s;
    }
    if (lane == 0) {
      sh.ival[0] = sg;
      sh.ival[1] = X | ((fb || fb2) ? 2 : 0);
      sh.scal[1] = rem2;
      sh.scal[2] = W;
      sh.scal[3] = W0;
    }
  }
  __syncthreads();
  const int sg = sh.ival[0];
  const int X = sh.ival[1] & 1;
  *zero = X != 0;
  *W_out = sh.scal[3];
  *near = true;
  if (sg < 0) return -1;
  const WProb wp{a.kT, wr.Mtk, wr.inv_st};
  // block `warp` of the segment: its sum
  const int g = sg * kSegBlocks + warp;
  stage_block1<E>(a, b, acc, g, warp, st);
  {
    const int i0 = (g * 32 + lane) * E::kVec;
    float ft[E::kVec], fd[E::kVec], x[E::kVec];
    E::unpack(st.fin.blk[warp][0][lane], ft);
    E::unpack(st.fin.blk[warp][1][lane], fd);
#pragma unroll
    for (int e = 0; e < E::kVec; ++e)
      x[e] = (i0 + e < a.V) ? (X ? wp(ft[e], 0.f, 0, 0.f) : wr(ft[e], fd[e], i0 + e, 0.f)) : 0.f;
    const float t = warp_incl_scan(lane_sum<E::kVec>(x));
    if (lane == 31) sh.bx[warp] = t;
  }
  __syncthreads();
  int bt = -1;
  if (warp == 0) {
    float rem3, W3;
    bool fb3;
    const int k = warp_locate(sh.bx, kSegBlocks, sh.scal[1], true, &rem3, &W3, &fb3);
    if (k >= 0) {
      const int gk = sg * kSegBlocks + k;
      const int i0 = (gk * 32 + lane) * E::kVec;
      float ft[E::kVec], fd[E::kVec], x[E::kVec];
      E::unpack(st.fin.blk[k][0][lane], ft);
      E::unpack(st.fin.blk[k][1][lane], fd);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e)
        x[e] = (i0 + e < a.V) ? (X ? wp(ft[e], 0.f, 0, 0.f) : wr(ft[e], fd[e], i0 + e, 0.f)) : 0.f;
      const float L = lane_sum<E::kVec>(x);
      const float incl = warp_incl_scan(L);
      float ex = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) ex = 0.f;
      float run = 0.f, edge = 0.f;
      int hit = -1, lpos = -1;
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) {
        const float before = __fadd_rn(ex, run);
        run = __fadd_rn(run, x[e]);
        if (x[e] > 0.f) {
          lpos = i0 + e;
          const float after = __fadd_rn(ex, run);
          if (hit < 0 && after > rem3) {
            hit = lpos;
            edge = fminf(__fsub_rn(rem3, before), __fsub_rn(after, rem3));
          }
        }
      }
      const uint32_t mc = __ballot_sync(0xffffffffu, L > 0.f && __fadd_rn(ex, L) > rem3);
      float dist = 0.f;
      if (mc) {
        const int src = __ffs(mc) - 1;
        dist = __shfl_sync(0xffffffffu, hit >= 0 ? fmaxf(edge, 0.f) : 0.f, src);
        bt = __shfl_sync(0xffffffffu, hit >= 0 ? hit : lpos, src);
      } else {
        bt = lpos;
#pragma unroll
        for (int o = 16; o; o >>= 1) bt = max(bt, __shfl_xor_sync(0xffffffffu, bt, o));
      }
      if (lane == 0) sh.ival[2] = ((sh.ival[1] & 2) || fb3 || bt < 0 || !(dist >= __fmul_rn(kNearTie, sh.scal[2]))) ? 1 : 0;
    } else if (lane == 0) {
      sh.ival[2] = 1;
    }
    if (lane == 0) sh.ival[3] = bt;
  }
  __syncthreads();
  *near = sh.ival[2] != 0;
  return sh.ival[3];
}

// Every thread: wait (bounded) for a ready word read by thread 0; when it does
// not come in time, for the completion of the whole pair grid instead.
SSD_DEV void await_word(const unsigned long long *w) {
  bool ok = true;
  if (threadIdx.x == 0) ok = wait_ready(w);
  if (__syncthreads_or(!ok)) asm volatile("griddepcontrol.wait;" ::: "memory");
}
// The lookup lists: the guess list of depth acc once its pair has written it
// (its ready word: thread 0 polls while the others load), and the payload,
// into `look` at their offsets when the lists are staged.
SSD_DEV void ready_lookup(const VocabArgs &a, int b, int acc, bool staged, int32_t *look) {
  if (!a.do_lookup) return;
  const int sumF = a.foff[a.K + 1];
  bool ok = true;
  if (threadIdx.x == 0) ok = wait_ready(&a.ready[(static_cast<size_t>(b) * (a.K + 1) + acc) * 2 + 1]);
  if (staged && a.payload && a.next_tokens)
    for (int i = threadIdx.x; i < sumF * a.K; i += kThreads)
      cp_async4(&look[sumF + i], a.payload + static_cast<size_t>(b) * sumF * a.K + i);
  if (__syncthreads_or(!ok)) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (staged)
    for (int i = threadIdx.x; i < a.F[acc]; i += kThreads)
      cp_async4(&look[a.foff[acc] + i], a.guess + static_cast<size_t>(b) * sumF + a.foff[acc] + i);
}
// The sequence's last unit (every thread): once the pair grid has completed no
// pair writes the sequence's ready words again; they go back to 0.
SSD_DEV void reset_ready(const VocabArgs &a, int b) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int t = threadIdx.x; t < 2 * a.npairs; t += kThreads)
    a.ready[static_cast<size_t>(b) * (a.K + 1) * 2 + t] = 0ull;
}

// 48 registers: every unit CTA then fits beside the pair kernel's CTAs, so no
// sequence's units wait for the pair grid to drain before they start.  CS: C < 1.
template <class E, bool CS>
__global__ void __maxnreg__(48) k_resid(const __grid_constant__ VocabArgs a) {
  __shared__ ResSh sh;
  extern __shared__ __align__(16) uint8_t res_smem[];
  ResStage &st = *reinterpret_cast<ResStage *>(res_smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = a.K;
  const int U = a.nunits;
  if (a.trace && tid == 0) {
    for (int k = 0; k < 8; ++k) sh.mk[k] = 0ull;
    sh.mk[1] = now_ns();
  }
  // verification waits for its own sequence's records (ready words); the
  // analytics for the whole pair grid
  // a statistics pass of the next (pipelined) call may start as soon as every
  // unit of this grid has started; nothing here waits for it
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const bool proto = a.ready != nullptr;
  if (!proto) asm volatile("griddepcontrol.wait;" ::: "memory");  // k_pair has completed
  int b = 0, u = 0;
  if (a.do_analytics) {
    // unit u of pair j < K (K = 0: one CTA per sequence, finishing it):
    // the sums of min(p, q') and of max(0, p - q')
    const int per = K > 0 ? K * U : 1;
    b = static_cast<int>(blockIdx.x) / per;
    const int rest = static_cast<int>(blockIdx.x) - b * per;
    const int j = K > 0 ? rest / U : 0;
    u = K > 0 ? rest - j * U : 0;
    int fin = K == 0 ? 1 : 0;
    if (K > 0) {
      float mn = 0.f, mx = 0.f;
      if (!a.greedy) {
        if (tid == 0) sh.rec[0] = a.rec[static_cast<size_t>(b) * (K + 1) + j];
        __syncthreads();
        const WResid wr = resid_weights(a, sh.rec[0], a.Fs[j]);
        unit_pass<E, true, CS>(a, b, j, u, wr, sh, st, &mn, &mx);
        __syncthreads();  // sh.seg is overwritten below
      }
      if (lane == 0) {
        sh.seg[warp][0] = mn;
        sh.seg[warp][1] = mx;
      }
      __syncthreads();
      if (tid == 0) {
        float m = 0.f, x = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          m = __fadd_rn(m, sh.seg[w][0]);
          x = __fadd_rn(x, sh.seg[w][1]);
        }
        a.amass[(static_cast<size_t>(b) * K + j) * U + u] = make_float2(m, x);
        __threadfence();
        if (atomicAdd(a.ctr + 2 + a.B + static_cast<size_t>(b) * K + j, 1u) + 1 == static_cast<uint32_t>(U)) {
          __threadfence();
          // alpha_j and W_j over the units in order; then this pair's ticket on the sequence
          if (!a.greedy) {
            float al = 0.f, W = 0.f;
            const float2 *src = a.amass + (static_cast<size_t>(b) * K + j) * U;
            for (int q = 0; q < U; ++q) {
              const float2 v = __ldcg(src + q);
              al = __fadd_rn(al, v.x);
              W = __fadd_rn(W, v.y);
            }
            PairRec *dst = a.rec + static_cast<size_t>(b) * (K + 1) + j;
            dst->al = al;
            dst->W = W;
          }
          __threadfence();
          fin = (atomicAdd(a.ctr + 2 + b, 1u) + 1 == static_cast<uint32_t>(K)) ? 1 : 0;
          if (fin) __threadfence();
        }
      }
    }
    if (tid == 0 && fin) {
      float run = 1.f, hit = 0.f, etok = 0.f;
      for (int k = 0; k <= K; ++k) {
        const PairRec *rp = a.rec + static_cast<size_t>(b) * (K + 1) + k;
        const float al = __ldcg(&rp->al), W = __ldcg(&rp->W), hp = __ldcg(&rp->hp), hr = __ldcg(&rp->hr);
        // the bonus given a = k follows r_{k+1} / W_{k+1} (p_{k+1} without residual mass), p_{K+1} for k = K
        const float h = (k < K && W > 0.f) ? __fdiv_rn(hr, W) : hp;
        const float pk = (k < K) ? __fmul_rn(run, W) : run;
        if (k < K) run = __fmul_rn(run, al);
        hit = __fmaf_rn(pk, h, hit);
        etok = __fmaf_rn(pk, static_cast<float>(k + 1), etok);
        a.an_p_accept[static_cast<size_t>(b) * (K + 1) + k] = pk;
        if (a.an_hit_mass) a.an_hit_mass[static_cast<size_t>(b) * (K + 1) + k] = h;
        if (k < K) {
          if (a.an_alpha) a.an_alpha[static_cast<size_t>(b) * K + k] = al;
          if (a.an_resid_w) a.an_resid_w[static_cast<size_t>(b) * K + k] = W;
        }
      }
      a.an_hit_rate[b] = hit;
      a.an_exp_tokens[b] = etok;
    }
  } else {
    // verification: the sequence's records and acceptance chain; its lookup
    // lists staged alongside (a finishing unit needs them)
    b = static_cast<int>(blockIdx.x) / U;
    u = static_cast<int>(blockIdx.x) - b * U;
    {  // verification calls always publish their records (ready words)
      bool ok = true;
      if (tid < a.npairs) ok = wait_ready(&a.ready[(static_cast<size_t>(b) * (K + 1) + tid) * 2]);
      if (__syncthreads_or(!ok)) asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    if (a.trace && tid == 0) sh.mk[2] = now_ns();
    const int sumF = a.foff[K + 1];
    const bool staged = a.do_lookup && sumF * (K + 1) <= kLookupStage;
    for (int i = tid; i < a.npairs * 4; i += kThreads)
      cp_async16(reinterpret_cast<int4 *>(sh.rec) + i, reinterpret_cast<const int4 *>(a.rec + static_cast<size_t>(b) * (K + 1)) + i);
    for (int t = tid; t < K; t += kThreads) sh.u[t] = a.u_acc[static_cast<size_t>(b) * K + t];
    cp_async_wait_all();
    __syncthreads();
    if (a.trace && tid == 0) sh.mk[3] = now_ns();
    int acc = 0;
    while (acc < K && (sh.rec[acc].fl & kRecAccepted)) ++acc;
    if (a.greedy || acc == K) {
      if (u == 0) {
        ready_lookup(a, b, acc, staged, st.fin.look);
        cp_async_wait_all();
        __syncthreads();
        const PairRec &r = sh.rec[acc];
        emit(a, b, acc, r.bt, r.W, (r.fl & kRecZero) != 0, (r.fl & kRecBonusNear) != 0, staged, sh,
             st.fin.look);
      }
      // every unit takes a ticket (a sole unit is the last); the last one resets the ready words
      if (tid == 0) {
        if (U == 1) {
          sh.ival[0] = 1;
        } else {
          __threadfence();
          sh.ival[0] = (atomicAdd(a.ctr + 2 + b, 1u) + 1 == static_cast<uint32_t>(U)) ? 1 : 0;
        }
      }
      __syncthreads();
      if (sh.ival[0]) reset_ready(a, b);
    } else {
      // the residual of the first rejected position: this unit's block sums
      const WResid wr = resid_weights(a, sh.rec[acc], a.Fs[acc]);
      float mn, mx;
      unit_pass<E, false, CS>(a, b, acc, u, wr, sh, st, &mn, &mx);
      __syncthreads();
      if (a.trace && tid == 0) sh.mk[4] = now_ns();
      if (warp == 0) {
        // the segment masses (two halves in order) and the unit's mass by
        // warp_runs' arithmetic over them
        const int nus = a.unit_sub * kResSeg;  // the unit's segments (<= 32), one per lane
        float vr = 0.f, vp = 0.f;
        if (lane < nus) {
          const int h = (lane / kResSeg) * kWarps + 2 * (lane % kResSeg);  // its first half in sh.seg
          vr = __fadd_rn(sh.seg[h][0], sh.seg[h + 1][0]);
          vp = __fadd_rn(sh.seg[h][1], sh.seg[h + 1][1]);
        }
        const int sg = u * nus + lane;
        if (lane < nus && sg < a.nseg) a.useg[static_cast<size_t>(b) * a.nseg + sg] = make_float2(vr, vp);
        const float ir = warp_incl_scan(vr);
        const float ip = warp_incl_scan(vp);
        if (U == 1) {
          // the sequence's sole unit is its last: its masses go straight to
          // where the draw reads them, without the round trip through memory
          if (lane < nus && sg < a.nseg) st.fin.sgm[sg] = make_float2(vr, vp);
          if (lane == 31) {
            sh.um[0][0] = ir;
            sh.um[1][0] = ip;
            sh.ival[0] = 1;
          }
        } else if (lane == 31) {
          a.umass[static_cast<size_t>(b) * U + u] = make_float2(ir, ip);
          __threadfence();
          const uint32_t t = atomicAdd(a.ctr + 2 + b, 1u);
          sh.ival[0] = (t + 1 == static_cast<uint32_t>(U)) ? 1 : 0;
          if (sh.ival[0]) __threadfence();
        }
      }
      __syncthreads();
      if (a.trace && tid == 0) sh.mk[5] = now_ns();
      if (sh.ival[0]) {
        // the last unit: the bonus.  Every unit and segment mass in one round
        // of loads while thread 0 checks that the outcome's guess list is
        // written; the lookup lists are copied while the draw runs.
        bool ok = true;
        if (tid == 0) {
          if (a.do_lookup) ok = wait_ready(&a.ready[(static_cast<size_t>(b) * (K + 1) + acc) * 2 + 1]);
        } else if (U > 1) {
          for (int q = tid - 1; q < U; q += kThreads - 1) {
            const float2 v = __ldcg(a.umass + static_cast<size_t>(b) * U + q);
            sh.um[0][q] = v.x;
            sh.um[1][q] = v.y;
          }
          for (int t = tid - 1; t < a.nseg; t += kThreads - 1)
            st.fin.sgm[t] = __ldcg(a.useg + static_cast<size_t>(b) * a.nseg + t);
        }
        if (staged && a.payload && a.next_tokens)
          for (int i = tid; i < sumF * K; i += kThreads)
            cp_async4(&st.fin.look[sumF + i], a.payload + static_cast<size_t>(b) * sumF * K + i);
        if (__syncthreads_or(!ok)) asm volatile("griddepcontrol.wait;" ::: "memory");
        if (staged)
          for (int i = tid; i < a.F[acc]; i += kThreads)
            cp_async4(&st.fin.look[a.foff[acc] + i], a.guess + static_cast<size_t>(b) * sumF + a.foff[acc] + i);
        float W;
        bool zero, near;
        int bt = resid_draw<E>(a, b, acc, wr, sh, st, &W, &zero, &near);
        if (bt < 0) {  // no weight at all: the target argmax
          bt = sh.rec[acc].bt;
          near = true;
        }
        if (a.trace && tid == 0) sh.mk[6] = now_ns();
        cp_async_wait_all();
        __syncthreads();
        emit(a, b, acc, bt, W, zero, near, staged, sh, st.fin.look);
        reset_ready(a, b);
      }
    }
  }
  if (a.trace && tid == 0) {
    sh.mk[7] = now_ns();
    trace_entry(a, a.trace_resid + blockIdx.x, 2, b, u, sh.mk);
  }
}

struct LookupArgs {
  const int32_t *guess, *payload, *accept_len, *bonus;
  int32_t *slot, *next_tokens;
  uint32_t *hits, *status;
  int B, K;
  int F[kMaxK + 1];
  int foff[kMaxK + 2];
};

__global__ void __launch_bounds__(256) k_lookup(const LookupArgs l) {
  __shared__ uint32_t tot;
  if (threadIdx.x == 0) tot = 0;
  __syncthreads();
  uint32_t h = 0;
  const int sumF = l.foff[l.K + 1];
  for (int b = threadIdx.x; b < l.B; b += blockDim.x) {
    const int acc = l.accept_len[b];
    int s = -1;
    if (acc < 0 || acc > l.K) {
      atomicOr(l.status, kFlagBadOutcome);
    } else {
      const int bt = l.bonus[b];
      for (int i = 0; i < l.F[acc]; ++i)
        if (l.guess[static_cast<size_t>(b) * sumF + l.foff[acc] + i] == bt) {
          s = l.foff[acc] + i;
          break;
        }
    }
    l.slot[b] = s;
    if (l.next_tokens)
      for (int t = 0; t < l.K; ++t)
        l.next_tokens[static_cast<size_t>(b) * l.K + t] =
            (s >= 0 && l.payload) ? l.payload[(static_cast<size_t>(b) * sumF + s) * l.K + t] : -1;
    h += (s >= 0);
  }
  atomicAdd(&tot, h);
  __syncthreads();
  if (threadIdx.x == 0 && l.hits) *l.hits = tot;
}

}  // namespace ssd

// ===========================================================================
// host side: validation, workspace layout, launches
// ===========================================================================
using namespace ssd;

namespace {

struct Layout {
  int nvec, nfull, nseg, nblk, nunits;
  size_t ctr_words, ctr_off, seg_off, bsum_off, bkey_off, rec_off, umass_off, useg_off, amass_off, ready_off, total;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int esize(ssd_dtype_t dt) { return dt == SSD_F32 ? 4 : 2; }

bool make_layout(int B, int K, int V, ssd_dtype_t dt, const int32_t *F, Layout *L) {
  if (B < 0 || K < 0 || K > kMaxK || V < 1 || !F) return false;
  if (dt != SSD_F32 && dt != SSD_BF16) return false;
  for (int k = 0; k <= K; ++k)
    if (F[k] < 0 || F[k] > kMaxF || F[k] > V) return false;
  const long long bytes = static_cast<long long>(V) * esize(dt);
  const long long nvec = (bytes + 15) / 16;
  const long long nseg = (nvec + kSegVec - 1) / kSegVec;
  if (nseg > kMaxSeg) return false;
  L->nvec = static_cast<int>(nvec);
  L->nfull = static_cast<int>(bytes / 16);
  L->nseg = static_cast<int>(nseg);
  L->nblk = L->nseg * kSegBlocks;
  L->nunits = (L->nseg + kResSeg - 1) / kResSeg;
  const size_t Bn = static_cast<size_t>(B > 0 ? B : 1);
  const size_t slots = Bn * 2 * (K + 1);
  L->ctr_words = 2 + Bn + Bn * K;
  size_t o = 0;
  L->ctr_off = o;
  o = align_up(o + L->ctr_words * sizeof(uint32_t), 256);
  L->seg_off = o;
  o = align_up(o + slots * L->nseg * sizeof(SegRec), 256);
  L->bsum_off = o;
  o = align_up(o + slots * L->nblk * sizeof(float), 256);
  L->bkey_off = o;
  o = align_up(o + slots * L->nblk * sizeof(uint32_t), 256);
  L->rec_off = o;
  o = align_up(o + Bn * (K + 1) * sizeof(PairRec), 256);
  L->umass_off = o;
  o = align_up(o + Bn * L->nunits * sizeof(float2), 256);
  L->useg_off = o;
  o = align_up(o + Bn * L->nseg * sizeof(float2), 256);
  L->amass_off = o;
  o = align_up(o + Bn * (K > 0 ? K : 1) * L->nunits * sizeof(float2), 256);
  L->ready_off = o;
  o = align_up(o + Bn * (K + 1) * 2 * sizeof(unsigned long long), 256);
  L->total = o;
  return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssd_status_t check_logits(const void *p, ssd_dtype_t dt, int64_t seq_stride, int64_t row_stride, int B, int K,
                          int V) {
  if (B == 0) return SSD_OK;
  if (!p) return SSD_ERR_INVALID_ARG;
  if (row_stride < V && K > 0) return SSD_ERR_INVALID_ARG;
  if (seq_stride < 0 || row_stride < 0) return SSD_ERR_INVALID_ARG;
  const int es = esize(dt);
  if (!aligned16(p) || (seq_stride * es) % 16 || (row_stride * es) % 16) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

ssd_status_t check_common(int B, float C, float T, const Layout &L, void *ws, size_t ws_bytes, bool needC) {
  if (!(T >= 0.f) || !isfinite(T)) return SSD_ERR_INVALID_ARG;
  if (needC && !(C > 0.f && C <= 1.f)) return SSD_ERR_INVALID_ARG;
  if (B > 0 && (!ws || ws_bytes < L.total)) return SSD_ERR_WORKSPACE;
  if (B > 0 && !aligned16(ws)) return SSD_ERR_INVALID_ARG;
  return SSD_OK;
}

ssd_status_t layout_or_error(int B, int K, int V, ssd_dtype_t dt, const int32_t *F, Layout *L) {
  if (!F || B < 0 || K < 0 || V < 1 || (dt != SSD_F32 && dt != SSD_BF16)) return SSD_ERR_INVALID_ARG;
  if (K > kMaxK) return SSD_ERR_UNSUPPORTED;
  for (int k = 0; k <= K; ++k)
    if (F[k] < 0) return SSD_ERR_INVALID_ARG;
  return make_layout(B, K, V, dt, F, L) ? SSD_OK : SSD_ERR_UNSUPPORTED;
}

VocabArgs base_args(const void *target, const void *draft, int64_t seq_stride, int64_t row_stride, int B, int K,
                    int V, const int32_t *F, float C, float T, const Layout &L, void *ws, uint32_t *status) {
  VocabArgs a;
  memset(&a, 0, sizeof(a));
  a.target = target;
  a.draft = draft;
  a.seq_stride = seq_stride;
  a.row_stride = row_stride;
  a.B = B;
  a.K = K;
  a.V = V;
  a.nvec = L.nvec;
  a.nfull = L.nfull;
  a.nseg = L.nseg;
  a.nblk = L.nblk;
  a.nunits = L.nunits;
  a.greedy = (T == 0.f);
  a.kT = a.greedy ? 0.f : static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  a.C = C;
  int off = 0;
  for (int k = 0; k <= K; ++k) {
    a.F[k] = F[k];
    a.foff[k] = off;
    off += F[k];
  }
  a.foff[K + 1] = off;
  char *w = static_cast<char *>(ws);
  a.ctr = reinterpret_cast<uint32_t *>(w + L.ctr_off);
  a.seg = reinterpret_cast<SegRec *>(w + L.seg_off);
  a.bsum = reinterpret_cast<float *>(w + L.bsum_off);
  a.bkey = reinterpret_cast<uint32_t *>(w + L.bkey_off);
  a.rec = reinterpret_cast<PairRec *>(w + L.rec_off);
  a.umass = reinterpret_cast<float2 *>(w + L.umass_off);
  a.useg = reinterpret_cast<float2 *>(w + L.useg_off);
  a.amass = reinterpret_cast<float2 *>(w + L.amass_off);
  a.ready = reinterpret_cast<unsigned long long *>(w + L.ready_off);
  a.status = status;
  return a;
}

// The device's SM count (queried once per device; 148 when it cannot be read).
int vocab_num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Rows read per position: target rows 0..ntarget-1 and draft rows 0..ndraft-1
// (slots ordered by pair: target j, then draft j); `topf`: the draft rows
// build their top-F_j lists.  Call after the do_* flags are set.
void set_rows(VocabArgs &a, int ntarget, int ndraft, bool topf) {
  a.npairs = ntarget > ndraft ? ntarget : ndraft;
  int n = 0;
  for (int j = 0; j <= a.K; ++j) {
    a.tsl[j] = a.dsl[j] = -1;
    a.Fs[j] = (topf && j < ndraft) ? a.F[j] : 0;
  }
  const bool draws = !a.greedy;
  for (int j = 0; j < a.npairs; ++j) {
    if (j < ntarget) {
      a.tsl[j] = n;
      // block sums on the rows a draw reads: target row K+1 (the bonus after
      // full acceptance) and the draft rows sampled from
      const bool blk = draws && a.do_verify && j == a.K;
      a.slot[n++] = RowSlot{0, static_cast<int16_t>(j), 0, static_cast<uint8_t>(blk), static_cast<uint8_t>(a.greedy),
                            0};
    }
    if (j < ndraft) {
      a.dsl[j] = n;
      const bool blk = draws && a.do_sample && j < a.K;
      a.slot[n++] = RowSlot{1, static_cast<int16_t>(j), static_cast<uint8_t>(a.Fs[j] >= 2), static_cast<uint8_t>(blk),
                            static_cast<uint8_t>(a.greedy || a.Fs[j] == 1), 0};
    }
  }
  a.nslots = n;
  a.unit_sub = 1;
  if (a.greedy) {
    a.nunits = 1;  // no residual pass: one finishing unit per sequence
  } else {
    // residual units of as many groups of kResSeg segments as keep the
    // residual grid near one wave of resident units (five per SM): small
    // batches keep one group per unit (the pass spread widest), large ones
    // fewer, fatter units (fewer waves, tickets and waits)
    const long groups = (a.nseg + kResSeg - 1) / kResSeg;
    const long per = a.do_analytics ? (a.K > 0 ? a.K : 1) : 1;
    const long work = static_cast<long>(a.B) * per * groups;
    // the analytics grid (every pair of every sequence) may take two waves
    const long slots = (a.do_analytics ? 10L : 5L) * vocab_num_sms();
    long sub = (work + slots - 1) / slots;
    if (sub > kMaxSub) sub = kMaxSub;
    if (sub > groups) sub = groups;
    if (sub < 1) sub = 1;
    // the same number of units with their groups spread evenly
    const long nu = (groups + sub - 1) / sub;
    sub = (groups + nu - 1) / nu;
    a.unit_sub = static_cast<int>(sub);
    a.nunits = static_cast<int>((groups + sub - 1) / sub);
  }
}

// Optional timing hook (ssd_set_timing_events): events recorded around the
// statistics kernel of every vocabulary call while set.
cudaEvent_t g_ev_before = nullptr;
cudaEvent_t g_ev_after = nullptr;
// Optional per-CTA trace (ssd_set_trace).
void *g_trace = nullptr;
size_t g_trace_bytes = 0;

ssd_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_attr_set[2][kMaxDevices / 64 + 1];

// A launch that may begin while the previous kernel on the stream drains
// (its CTAs wait for that kernel with griddepcontrol.wait).
template <class Kern>
cudaError_t launch_dependent(Kern kern, unsigned grid, size_t smem, cudaStream_t s, const VocabArgs &a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// k_stats over every (chunk of 4 segments, row slot, sequence), then k_pair
// (one CTA per sequence and row pair) and, when verifying or for the
// analytics, k_resid.
template <class E>
cudaError_t launch_vocab(VocabArgs &a, cudaStream_t s) {
  constexpr int ti = E::kSize == 4 ? 0 : 1;
  if (a.B < 1 || a.npairs < 1) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const size_t psmem = pair_smem_bytes(a.nseg, a.nblk);
  const uint64_t bit = 1ull << (dev % 64);
  if (!(g_attr_set[ti][dev / 64].load() & bit)) {
    e = cudaFuncSetAttribute(k_pair<E, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(pair_smem_bytes(kMaxSeg, kMaxSeg * kSegBlocks)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_pair<E, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(pair_smem_bytes(kMaxSeg, kMaxSeg * kSegBlocks)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_resid<E, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sizeof(ResStage)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_resid<E, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sizeof(ResStage)));
    if (e != cudaSuccess) return e;
    g_attr_set[ti][dev / 64].fetch_or(bit);
  }
  const unsigned nchunks = static_cast<unsigned>((a.nseg + kStatWarps - 1) / kStatWarps);
  const long n1 = static_cast<long>(nchunks) * a.nslots * a.B;
  const long n2 = static_cast<long>(a.B) * a.npairs;
  const bool resid = a.do_verify || a.do_analytics;
  const long n3 = !resid ? 0 : (a.do_analytics ? static_cast<long>(a.B) * (a.K > 0 ? a.K * a.nunits : 1)
                                               : static_cast<long>(a.B) * a.nunits);
  if (n2 > 0x7fffffffL || n3 > 0x7fffffffL) return cudaErrorInvalidValue;
  a.trace = (g_trace && a.B <= 65535 && g_trace_bytes >= static_cast<size_t>(n1 + n2 + n3) * 64)
                ? static_cast<unsigned long long *>(g_trace)
                : nullptr;
  a.trace_pair = n1;
  a.trace_resid = n1 + n2;
  if (!(a.do_verify && !a.do_analytics)) a.ready = nullptr;
  if (g_ev_before) cudaEventRecord(g_ev_before, s);
  // grid (chunk, row slot, sequence); sequences in launches of at most 65535
  for (int b0 = 0; b0 < a.B; b0 += 65535) {
    a.b0 = b0;
    const unsigned nb = static_cast<unsigned>(a.B - b0 < 65535 ? a.B - b0 : 65535);
    const dim3 grid(nchunks, static_cast<unsigned>(a.nslots), nb);
    if (a.pipelined && b0 == 0) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = grid;
      cfg.blockDim = dim3(kStatWarps * 32);
      cfg.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, k_stats<E>, a);
    } else {
      k_stats<E><<<grid, kStatWarps * 32, 0, s>>>(a);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  a.b0 = 0;
  if (g_ev_after) cudaEventRecord(g_ev_after, s);
  e = launch_dependent(a.C < 1.f ? k_pair<E, true> : k_pair<E, false>, static_cast<unsigned>(n2), psmem, s, a);
  if (e != cudaSuccess || n3 == 0) return e;
  return launch_dependent(a.C < 1.f ? k_resid<E, true> : k_resid<E, false>, static_cast<unsigned>(n3), sizeof(ResStage), s,
                          a);
}

cudaError_t launch_any(ssd_dtype_t dt, VocabArgs &a, cudaStream_t s) {
  return dt == SSD_F32 ? launch_vocab<EF32>(a, s) : launch_vocab<EBF16>(a, s);
}

// Fixed device scratch for ssd_verify_noalloc: one array per GPU that loads
// the library, held until the process exits.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

void *g_static_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_static_scratch_mu;

// Device address of g_static_scratch on the current device, looked up once per
// device (the array's name in host code is only a stand-in for it).
cudaError_t static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (!g_static_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

const char *ssd_status_string(ssd_status_t st) {
  switch (st) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case SSD_ERR_WORKSPACE: return "workspace missing or too small";
    case SSD_ERR_CUDA: return "CUDA launch error";
  }
  return "unknown status";
}

ssd_status_t ssd_fanout_split(int budget, int K, double r, int32_t *F_out) {
  if (!F_out || K < 0 || K > kMaxK || budget < K + 1 || !(r > 0.0) || r > 1.0) return SSD_ERR_INVALID_ARG;
  double w[kMaxK + 1], sw = 0.0, frac[kMaxK + 1];
  double rk = 1.0;
  for (int k = 0; k <= K; ++k) {
    w[k] = rk;
    sw += rk;
    rk *= r;
  }
  int total = 0;
  for (int k = 0; k <= K; ++k) {
    const double x = budget * w[k] / sw;
    const double fl = floor(x);
    frac[k] = x - fl;
    F_out[k] = static_cast<int32_t>(fl) < 1 ? 1 : static_cast<int32_t>(fl);
    total += F_out[k];
  }
  // hand out a shortfall by descending fractional part (ties: smaller k)
  bool used[kMaxK + 1] = {false};
  while (total < budget) {
    int best = -1;
    for (int k = 0; k <= K; ++k)
      if (!used[k] && (best < 0 || frac[k] > frac[best])) best = k;
    if (best < 0) {
      for (int k = 0; k <= K; ++k) used[k] = false;
      continue;
    }
    used[best] = true;
    ++F_out[best];
    ++total;
  }
  // take an excess from the largest F_k > 1 (ties: larger k)
  while (total > budget) {
    int best = -1;
    for (int k = 0; k <= K; ++k)
      if (F_out[k] > 1 && (best < 0 || F_out[k] >= F_out[best])) best = k;
    if (best < 0) return SSD_ERR_INVALID_ARG;
    --F_out[best];
    --total;
  }
  return SSD_OK;
}

ssd_status_t ssd_set_timing_events(void *before, void *after) {
  if ((before == nullptr) != (after == nullptr)) return SSD_ERR_INVALID_ARG;
  g_ev_before = static_cast<cudaEvent_t>(before);
  g_ev_after = static_cast<cudaEvent_t>(after);
  return SSD_OK;
}

ssd_status_t ssd_set_trace(void *buf, size_t bytes) {
  g_trace = buf;
  g_trace_bytes = buf ? bytes : 0;
  return SSD_OK;
}

size_t ssd_workspace_size(int B, int K, int V, ssd_dtype_t dt, const int32_t *F) {
  Layout L;
  if (!make_layout(B, K, V, dt, F, &L)) return 0;
  return L.total;
}

ssd_status_t ssd_saguaro_sample(const void *draft, ssd_dtype_t dt, int64_t seq_stride, int64_t row_stride,
                                int B, int K, int V, const int32_t *F, float C, float T, const float *u_draft,
                                int32_t *d_out, float *qd_out, uint32_t *status, void *ws, size_t ws_bytes,
                                ssd_stream_t s) {
  Layout L;
  ssd_status_t st = layout_or_error(B, K, V, dt, F, &L);
  if (st != SSD_OK) return st;
  st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(B, C, T, L, ws, ws_bytes, true);
  if (st != SSD_OK) return st;
  if (B == 0 || K == 0) return SSD_OK;
  if (!u_draft || !d_out || !status) return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(draft, draft, seq_stride, row_stride, B, K, V, F, C, T, L, ws, status);
  a.do_sample = 1;
  set_rows(a, 0, K, C < 1.f);
  a.u_draft = u_draft;
  a.d_out = d_out;
  a.qd_out = qd_out;
  return cuda_status(launch_any(dt, a, reinterpret_cast<cudaStream_t>(s)));
}

ssd_status_t ssd_fill_sample(const void *logits, ssd_dtype_t dt, int64_t branch_stride, int B, int S, int V,
                             int F_t, float C, float T, const float *u, int t, int Kp, int32_t *tokens,
                             float *q_out, int32_t *payload, uint32_t *status, void *ws, size_t ws_bytes,
                             ssd_stream_t s) {
  // every branch row is a one-draw "sequence": K = 1, F = (F_t, 0)
  if (B < 0 || S < 0 || (payload && (Kp < 1 || t < 0 || t >= Kp))) return SSD_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * S;
  if (rows > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
  const int32_t F[2] = {F_t, 0};
  const int Bp = static_cast<int>(rows);
  Layout L;
  ssd_status_t st = layout_or_error(Bp, 1, V, dt, F, &L);
  if (st != SSD_OK) return st;
  st = check_logits(logits, dt, branch_stride, branch_stride, Bp, 1, V);
  if (st != SSD_OK) return st;
  st = check_common(Bp, C, T, L, ws, ws_bytes, true);
  if (st != SSD_OK) return st;
  if (Bp == 0) return SSD_OK;
  if (!u || !tokens || !status) return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(logits, logits, branch_stride, branch_stride, Bp, 1, V, F, C, T, L, ws, status);
  a.do_sample = 1;
  set_rows(a, 0, 1, C < 1.f);
  a.u_draft = u;
  a.d_out = tokens;
  a.qd_out = q_out;
  a.fill_payload = payload;
  a.fill_stride = Kp;
  a.fill_col = t;
  return cuda_status(launch_any(dt, a, reinterpret_cast<cudaStream_t>(s)));
}

ssd_status_t ssd_verify(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                        int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                        const int32_t *d, const float *u_acc, const float *u_bonus, int32_t *accept_len,
                        int32_t *out_tokens, int32_t *bonus, float *accept_prob, float *resid_mass,
                        uint32_t *near_ties, uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s) {
  Layout L;
  ssd_status_t st = layout_or_error(B, K, V, dt, F, &L);
  if (st != SSD_OK) return st;
  st = check_logits(target, dt, seq_stride, row_stride, B, K, V);
  if (st == SSD_OK) st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(B, C, T, L, ws, ws_bytes, true);
  if (st != SSD_OK) return st;
  if (B == 0) return SSD_OK;
  if ((K > 0 && (!d || !u_acc)) || !u_bonus || !accept_len || !out_tokens || !bonus || !status)
    return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(target, draft, seq_stride, row_stride, B, K, V, F, C, T, L, ws, status);
  a.do_verify = 1;
  set_rows(a, K + 1, K, C < 1.f);
  a.d_in = d;
  a.u_acc = u_acc;
  a.u_bonus = u_bonus;
  a.accept_len = accept_len;
  a.out_tokens = out_tokens;
  a.bonus = bonus;
  a.accept_prob = accept_prob;
  a.resid_mass = resid_mass;
  a.near_ties = near_ties;
  return cuda_status(launch_any(dt, a, reinterpret_cast<cudaStream_t>(s)));
}

ssd_status_t ssd_predict_outcomes(const void *draft, ssd_dtype_t dt, int64_t seq_stride, int64_t row_stride,
                                  int B, int K, int V, const int32_t *F, float T, int32_t *guess, float *guess_q,
                                  uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s) {
  Layout L;
  ssd_status_t st = layout_or_error(B, K, V, dt, F, &L);
  if (st != SSD_OK) return st;
  st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(B, 1.f, T, L, ws, ws_bytes, false);
  if (st != SSD_OK) return st;
  if (B == 0) return SSD_OK;
  if (!guess || !status) return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(draft, draft, seq_stride, row_stride, B, K, V, F, 1.f, T, L, ws, status);
  a.do_predict = 1;
  set_rows(a, 0, K + 1, true);
  a.guess = guess;
  a.guess_q = guess_q;
  return cuda_status(launch_any(dt, a, reinterpret_cast<cudaStream_t>(s)));
}

ssd_status_t ssd_cache_lookup(const int32_t *guess, const int32_t *payload, int B, int K, const int32_t *F,
                              const int32_t *accept_len, const int32_t *bonus, int32_t *slot,
                              int32_t *next_tokens, uint32_t *hits, uint32_t *status, ssd_stream_t s) {
  if (B < 0 || K < 0 || K > kMaxK || !F) return SSD_ERR_INVALID_ARG;
  for (int k = 0; k <= K; ++k)
    if (F[k] < 0 || F[k] > kMaxF) return SSD_ERR_INVALID_ARG;
  if (B == 0) {
    if (hits) return cuda_status(cudaMemsetAsync(hits, 0, sizeof(uint32_t), reinterpret_cast<cudaStream_t>(s)));
    return SSD_OK;
  }
  if (!guess || !accept_len || !bonus || !slot || !status) return SSD_ERR_INVALID_ARG;
  LookupArgs l;
  memset(&l, 0, sizeof(l));
  l.guess = guess;
  l.payload = payload;
  l.accept_len = accept_len;
  l.bonus = bonus;
  l.slot = slot;
  l.next_tokens = next_tokens;
  l.hits = hits;
  l.status = status;
  l.B = B;
  l.K = K;
  int off = 0;
  for (int k = 0; k <= K; ++k) {
    l.F[k] = F[k];
    l.foff[k] = off;
    off += F[k];
  }
  l.foff[K + 1] = off;
  k_lookup<<<1, 256, 0, reinterpret_cast<cudaStream_t>(s)>>>(l);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"

namespace {
ssd_status_t round_impl(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                        int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                        const float *u_draft, const float *u_acc, const float *u_bonus, const int32_t *payload,
                        int32_t *d_out, float *qd_out, int32_t *accept_len, int32_t *out_tokens, int32_t *bonus,
                        float *accept_prob, float *resid_mass, int32_t *guess, float *guess_q, int32_t *slot,
                        int32_t *next_tokens, uint32_t *hits, uint32_t *near_ties, uint32_t *status, void *ws,
                        size_t ws_bytes, ssd_stream_t s, bool pipelined) {
  Layout L;
  ssd_status_t st = layout_or_error(B, K, V, dt, F, &L);
  if (st != SSD_OK) return st;
  st = check_logits(target, dt, seq_stride, row_stride, B, K, V);
  if (st == SSD_OK) st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(B, C, T, L, ws, ws_bytes, true);
  if (st != SSD_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  if (B == 0) {
    if (hits) return cuda_status(cudaMemsetAsync(hits, 0, sizeof(uint32_t), cs));
    return SSD_OK;
  }
  if ((K > 0 && (!u_draft || !u_acc || !d_out)) || !u_bonus || !accept_len || !out_tokens || !bonus || !status)
    return SSD_ERR_INVALID_ARG;
  if ((slot || next_tokens || hits) && !guess) return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(target, draft, seq_stride, row_stride, B, K, V, F, C, T, L, ws, status);
  a.do_sample = 1;
  a.do_verify = 1;
  a.do_predict = guess != nullptr;
  a.do_lookup = guess != nullptr;
  set_rows(a, K + 1, a.do_predict ? K + 1 : K, a.do_predict || C < 1.f);
  a.u_draft = u_draft;
  a.u_acc = u_acc;
  a.u_bonus = u_bonus;
  a.payload = payload;
  a.d_out = d_out;
  a.qd_out = qd_out;
  a.accept_len = accept_len;
  a.out_tokens = out_tokens;
  a.bonus = bonus;
  a.accept_prob = accept_prob;
  a.resid_mass = resid_mass;
  a.guess = guess;
  a.guess_q = guess_q;
  a.slot_out = slot;
  a.next_tokens = next_tokens;
  a.hits = hits;
  a.near_ties = near_ties;
  a.pipelined = pipelined ? 1 : 0;
  return cuda_status(launch_any(dt, a, cs));
}
}  // namespace

extern "C" {

ssd_status_t ssd_round(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                       int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                       const float *u_draft, const float *u_acc, const float *u_bonus, const int32_t *payload,
                       int32_t *d_out, float *qd_out, int32_t *accept_len, int32_t *out_tokens, int32_t *bonus,
                       float *accept_prob, float *resid_mass, int32_t *guess, float *guess_q, int32_t *slot,
                       int32_t *next_tokens, uint32_t *hits, uint32_t *near_ties, uint32_t *status, void *ws,
                       size_t ws_bytes, ssd_stream_t s) {
  return round_impl(target, draft, dt, seq_stride, row_stride, B, K, V, F, C, T, u_draft, u_acc, u_bonus, payload,
                    d_out, qd_out, accept_len, out_tokens, bonus, accept_prob, resid_mass, guess, guess_q, slot,
                    next_tokens, hits, near_ties, status, ws, ws_bytes, s, false);
}

ssd_status_t ssd_round_pipelined(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                                 int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                                 const float *u_draft, const float *u_acc, const float *u_bonus,
                                 const int32_t *payload, int32_t *d_out, float *qd_out, int32_t *accept_len,
                                 int32_t *out_tokens, int32_t *bonus, float *accept_prob, float *resid_mass,
                                 int32_t *guess, float *guess_q, int32_t *slot, int32_t *next_tokens,
                                 uint32_t *hits, uint32_t *near_ties, uint32_t *status, void *ws, size_t ws_bytes,
                                 ssd_stream_t s) {
  return round_impl(target, draft, dt, seq_stride, row_stride, B, K, V, F, C, T, u_draft, u_acc, u_bonus, payload,
                    d_out, qd_out, accept_len, out_tokens, bonus, accept_prob, resid_mass, guess, guess_q, slot,
                    next_tokens, hits, near_ties, status, ws, ws_bytes, s, true);
}

ssd_status_t ssd_round_analytics(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                                 int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                                 float *alpha, float *resid_w, float *p_accept, float *hit_mass, float *hit_rate,
                                 float *exp_tokens, uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s) {
  Layout L;
  ssd_status_t st = layout_or_error(B, K, V, dt, F, &L);
  if (st != SSD_OK) return st;
  st = check_logits(target, dt, seq_stride, row_stride, B, K, V);
  if (st == SSD_OK) st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(B, C, T, L, ws, ws_bytes, true);
  if (st != SSD_OK) return st;
  if (B == 0) return SSD_OK;
  if (!p_accept || !hit_rate || !exp_tokens || !status) return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(target, draft, seq_stride, row_stride, B, K, V, F, C, T, L, ws, status);
  a.do_analytics = 1;
  set_rows(a, K + 1, K + 1, true);
  a.an_alpha = alpha;
  a.an_resid_w = resid_w;
  a.an_p_accept = p_accept;
  a.an_hit_mass = hit_mass;
  a.an_hit_rate = hit_rate;
  a.an_exp_tokens = exp_tokens;
  return cuda_status(launch_any(dt, a, reinterpret_cast<cudaStream_t>(s)));
}

size_t ssd_verify_noalloc_max_bytes(void) { return kStaticScratchBytes; }

ssd_status_t ssd_verify_noalloc(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                                int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                                const int32_t *d, const float *u_acc, const float *u_bonus,
                                int32_t *accept_len, int32_t *out_tokens, int32_t *bonus, float *accept_prob,
                                float *resid_mass, uint32_t *near_ties, uint32_t *status, ssd_stream_t s) {
  // every argument error maps as in ssd_verify; only then the scratch size
  Layout L;
  ssd_status_t st = layout_or_error(B, K, V, dt, F, &L);
  if (st != SSD_OK) return st;
  st = check_logits(target, dt, seq_stride, row_stride, B, K, V);
  if (st == SSD_OK) st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  if (!(T >= 0.f) || !isfinite(T) || !(C > 0.f && C <= 1.f)) return SSD_ERR_INVALID_ARG;
  if (B == 0) return SSD_OK;
  if ((K > 0 && (!d || !u_acc)) || !u_bonus || !accept_len || !out_tokens || !bonus || !status)
    return SSD_ERR_INVALID_ARG;
  if (L.total > kStaticScratchBytes) return SSD_ERR_WORKSPACE;  // the batch needs more scratch than the array holds
  void *ws = nullptr;
  if (static_scratch(&ws) != cudaSuccess) return SSD_ERR_CUDA;
  return ssd_verify(target, draft, dt, seq_stride, row_stride, B, K, V, F, C, T, d, u_acc, u_bonus, accept_len,
                    out_tokens, bonus, accept_prob, resid_mass, near_ties, status, ws, kStaticScratchBytes, s);
}

}  // extern "C"
