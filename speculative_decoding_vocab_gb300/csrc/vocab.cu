// vocab.cu -- the vocabulary-wide kernels of one speculation round on sm_103a:
// Saguaro draft sampling, lossless verification with residual / bonus draw,
// outcome prediction (top-F_k guesses) and the speculation-cache lookup.
//
// Method: speculative-speculative decoding with the Saguaro algorithm as the
// 機器之心 article "全球最強推理引擎還快2倍，斯坦福、普林斯頓破解大模型串行魔咒"
// (section "SSD 如何實現草擬與驗證并行？") and the technical summary
// "超越传统SD：SSD框架全异步解码实现4.7倍平均加速" (sections "投机解码的瓶颈与 SSD 的
// 核心机制" and "Saguaro 算法" parts 1-2) describe it; the readings of the
// missing formulas are stated in include/ssd.h at each call.
//
// Structure: a vocabulary call is at most two kernels.
//   k_stats  one CTA per 32 KiB chunk of one logit row: the HBM pass, which
//            carries nearly all of the call's bytes.  A TMA bulk copy stages
//            the chunk in shared memory; the CTA reduces it to a record (max,
//            sum of 2^(z log2e/T - max), argmax), per-block partial sums for
//            rows that are drawn from (a block = the 32 vectors one warp reads
//            in one round) and per-block maximum keys for rows with a top-F
//            list.  Chunks are numbered sequence-major and, within a sequence,
//            by row pair r = (target row r, draft row r).  Each CTA takes its
//            pair's ticket while its copy is in flight: the last CTA of a pair
//            to start merges the pair once the others are published (row
//            statistics, the top-F_r list from the block maxima, the Saguaro
//            draw of d_{r+1}, p(d) and q'(d), the position's verdict), and the
//            last merger of a sequence to start runs the acceptance chain and,
//            unless a residual draw is needed, the bonus draw and the outputs.
//            A merger waits only for CTAs that started before it.  A draw
//            locates its chunk from the chunk masses and its block from the
//            block sums; one warp then reads that block's 32 vectors again.
//            The merges stage the records they read in shared memory (over
//            the chunk buffer) with one round of loads.
//   k_resid  (verification at T > 0) one CTA per quarter chunk of each
//            sequence's rejected row pair: residual block sums; the unit with
//            the sequence's last ticket draws the bonus token from them and
//            writes the outputs.  It is a programmatic dependent launch of
//            k_stats: its CTAs start once every k_stats CTA has started, and
//            each waits only for its own sequence's ready word, which the pair
//            merges set as soon as the first rejected position is known.
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
constexpr int kStatsCtas = 5;  // resident k_stats CTAs per SM
constexpr int kWarps = kThreads / 32;
constexpr int kRounds = 8;                             // 16-byte vectors per thread and chunk
constexpr int kChunkBytes = kThreads * kRounds * 16;  // 32 KiB
constexpr int kBlocks = kRounds * kWarps;              // blocks per chunk (round j, warp w)
constexpr int kQuarters = 4;                           // k_resid units per chunk (2 rounds each)
constexpr int kCandCap = 512;
constexpr int kMaxK = 16;
constexpr int kMaxSlots = 2 * (kMaxK + 1);
constexpr int kMaxF = 256;
constexpr int kMaxChunks = 128;  // per row: 4 chunk records per lane in the warp merge
constexpr int kNone = 0x7fffffff;
// A draw whose target lies within kNearTie * W of an edge of the chosen
// element's bin, and an acceptance test with |u - p/q'| < kNearTie, is a
// near-tie: fp32 and exact arithmetic may decide it differently.  Such
// events are counted (the optional near_ties output).
constexpr float kNearTie = 1e-6f;

struct __align__(16) ChunkStat {
  float m;   // chunk maximum
  float s;   // sum over the chunk of 2^(z kT - fl(m kT)) (0 when greedy)
  int amax;  // lowest index holding m
  int pad;
};
// Per chunk of a row that is drawn from: each warp's maximum and, per block
// (round j, warp w), the sum of 2^(z kT - fl(wm[w] kT)) over the block's
// elements (0 when greedy or for a warp without finite elements).
struct __align__(16) BlockRec {
  float wm[kWarps];
  float bs[kRounds][kWarps];
};
struct RowSlot {
  int16_t tensor;  // 0 = target, 1 = draft
  int16_t row;
  int16_t F;       // top-F candidates wanted (0 = none)
  int16_t blocks;  // block sums wanted (the row is drawn from)
};
struct __align__(16) RowInfo {  // merged statistics of row r of a sequence
  float mt, st;   // target max, sum relative to fl(mt kT)
  int at, pad0;   // target argmax
  float md, sd;   // draft max, sum
  int ad;         // draft argmax
  float sq;       // sum of q over S (normalised)
};
struct __align__(16) PosInfo {  // draft token d_j and its probabilities
  int d;
  float p, q;  // p_j(d), q'_j(d); p < 0 marks an invalid token
  int pad;
};

struct VocabArgs {
  const void *target, *draft;
  int64_t seq_stride, row_stride;  // elements
  int B, K, V;
  int nslots, nchunks, chunk_elems, Fcap;
  float kT;    // log2(e) / T
  int greedy;  // T == 0
  float C;
  int npairs;  // row pairs per sequence, r = 0 .. npairs-1
  long nst;    // chunks of the call: B * nslots * nchunks
  int b0;      // k_stats: the first sequence of this launch (grid z = sequence - b0)
  int do_sample, do_verify, do_predict, do_lookup, do_analytics;
  RowSlot slot[kMaxSlots];                   // ordered by pair: target r, then draft r
  int tsl[kMaxK + 1], dsl[kMaxK + 1];        // slot of target / draft row r (-1: none)
  int pair_chunks[kMaxK + 1];                // chunks of pair r (both rows)
  int F[kMaxK + 1];                          // fan-out F_r
  int Fs[kMaxK + 1];                         // top-F list kept for draft row r (F_r or 0)
  int foff[kMaxK + 2];
  // workspace
  uint32_t *ctr;  // [0] finished sequences, [1] hits; per sequence b: [2+b] pair-merge
                  // tickets, [2+B+b] merged pairs published, [2+2B+b] residual unit
                  // tickets, [2+3B+b] ready word (accept count + 2 once known),
                  // [2+4B+b] residual units published; per pair (b, r):
                  // [2+5B + b(K+1)+r] chunk tickets, [2+5B+B(K+1) + b(K+1)+r]
                  // chunks published, [2+5B+2B(K+1) + b(K+1)+r] position verdict
  ChunkStat *stats;  // [B][nslots][nchunks]
  BlockRec *blk;     // [B][nslots][nchunks]
  uint32_t *bmk;     // [B][nslots][nchunks][kBlocks] block maximum keys of top-F rows (0: empty block)
  RowInfo *rows;     // [B][K+1]
  uint64_t *S;       // [B][K+1][Fcap] merged top-F lists
  PosInfo *pos;      // [B][K]
  float *rmass;      // [B][nchunks * kQuarters] residual mass per unit
  float *rbs;        // [B][nchunks][kBlocks] residual block sums
  float *amass;      // analytics: [B][K][nchunks * kQuarters][2] unit sums of min(p, q'), max(0, p - q')
  // analytics outputs
  float *an_alpha, *an_resid_w, *an_p_accept, *an_hit_mass, *an_hit_rate, *an_exp_tokens;
  // inputs / outputs
  const float *u_draft, *u_acc, *u_bonus;
  const int32_t *d_in;
  const int32_t *payload;
  int32_t *d_out;
  float *qd_out;
  int32_t *accept_len, *out_tokens, *bonus;
  float *accept_prob, *resid_mass;
  int32_t *guess;
  float *guess_q;
  int32_t *slot_out, *next_tokens;
  uint32_t *hits;
  uint32_t *near_ties;  // optional: near-tie draws and tests, added to
  uint32_t *status;
  unsigned long long *trace;  // optional: 8 words per CTA (see ssd_set_trace)
};

SSD_DEV uint32_t *seq_tkt(const VocabArgs &a, int b) { return a.ctr + 2 + b; }
SSD_DEV uint32_t *seq_pub(const VocabArgs &a, int b) { return a.ctr + 2 + a.B + b; }
SSD_DEV uint32_t *res_tkt(const VocabArgs &a, int b) { return a.ctr + 2 + 2 * a.B + b; }
SSD_DEV uint32_t *ready_word(const VocabArgs &a, int b) { return a.ctr + 2 + 3 * a.B + b; }
SSD_DEV uint32_t *res_pub(const VocabArgs &a, int b) { return a.ctr + 2 + 4 * a.B + b; }
SSD_DEV uint32_t *pair_tkt(const VocabArgs &a, int b, int r) {
  return a.ctr + 2 + 5 * static_cast<size_t>(a.B) + static_cast<size_t>(b) * (a.K + 1) + r;
}
SSD_DEV uint32_t *pair_pub(const VocabArgs &a, int b, int r) {
  return pair_tkt(a, b, r) + static_cast<size_t>(a.B) * (a.K + 1);
}
// Verification of position r of sequence b, once its pair is merged: 1
// accepted, 2 rejected (0: not yet known).
SSD_DEV uint32_t *pos_verdict(const VocabArgs &a, int b, int r) {
  return pair_tkt(a, b, r) + 2 * static_cast<size_t>(a.B) * (a.K + 1);
}
__host__ __device__ inline size_t ctr_words(size_t B, int K) { return 2 + 5 * B + 3 * B * (K + 1); }

__host__ __device__ inline size_t chunk_index(const VocabArgs &a, int b, int slot, int c) {
  return (static_cast<size_t>(b) * a.nslots + slot) * a.nchunks + c;
}
SSD_DEV const char *row_ptr(const VocabArgs &a, int tensor, int b, int row, int esize) {
  const char *base = reinterpret_cast<const char *>(tensor ? a.draft : a.target);
  return base + (static_cast<int64_t>(b) * a.seq_stride + static_cast<int64_t>(row) * a.row_stride) * esize;
}

// ---------------------------------------------------------------------------
// loads of records other CTAs published (L2, never a stale L1 line)
// ---------------------------------------------------------------------------
SSD_DEV ChunkStat ldcg_stat(const ChunkStat *p) {
  const int4 v = __ldcg(reinterpret_cast<const int4 *>(p));
  return ChunkStat{__int_as_float(v.x), __int_as_float(v.y), v.z, v.w};
}
SSD_DEV RowInfo ldcg_row(const RowInfo *p) {
  const int4 v = __ldcg(reinterpret_cast<const int4 *>(p));
  const int4 w = __ldcg(reinterpret_cast<const int4 *>(p) + 1);
  return RowInfo{__int_as_float(v.x), __int_as_float(v.y), v.z,    v.w,
                 __int_as_float(w.x), __int_as_float(w.y), w.z, __int_as_float(w.w)};
}
SSD_DEV PosInfo ldcg_pos(const PosInfo *p) {
  const int4 v = __ldcg(reinterpret_cast<const int4 *>(p));
  return PosInfo{v.x, __int_as_float(v.y), __int_as_float(v.z), v.w};
}
SSD_DEV uint64_t ldcg_key(const uint64_t *p) { return __ldcg(reinterpret_cast<const unsigned long long *>(p)); }

// Arrivals and polls are release / relaxed; only the CTA that goes on to read
// what others published pays for the acquire (a fence), since an acquire
// invalidates the SM's L1, where the other resident CTAs keep their spills.
SSD_DEV uint32_t ld_relaxed(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
SSD_DEV void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
SSD_DEV uint32_t atom_add_release(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
SSD_DEV void red_add_release(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
SSD_DEV void st_release(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Trace mark k of this CTA (ssd_set_trace): %globaltimer by thread 0.
SSD_DEV void mark(const VocabArgs &a, unsigned long long *mk, int k) {
  if (a.trace && threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    mk[k] = t;
  }
}

// ---------------------------------------------------------------------------
// shared memory of a CTA (k_stats: after the staged chunk)
// ---------------------------------------------------------------------------
struct Smem {
  uint64_t bar;  // k_stats: completion of the chunk's TMA copy
  int flag, ncand;
  alignas(16) uint32_t hist[2][256];  // top-F threshold: block maxima counted by key byte (read as 16-byte vectors)
  float wm[kWarps], ws[kWarps];
  int wa[kWarps];
  uint64_t redk[kWarps];
  float scal[8];
  int ival[8];
  RowInfo ri;
  uint64_t cand[kCandCap];  // pair merge: candidate block list; sequence finish: the lookup's lists
  float cmass[kMaxChunks];
  float bw[kBlocks];
  uint64_t S[kMaxF];
  PosInfo pos[kMaxK];  // draft tokens, p(d), q'(d)
  float cu[kMaxK];     // acceptance uniforms
  RowInfo rows[kMaxK + 1];
  uint64_t keyF[kMaxK + 1];
  unsigned long long mk[7];  // trace marks (thread 0)
  int near;                  // thread 0: the last draw was a near-tie (its target within 1e-6 W of a bin edge)
};

// What a merge reads of other CTAs' records, staged in shared memory by one
// round of loads (k_stats: laid over the chunk buffer once the chunk's own
// statistics are published).
constexpr int kStageChunks = 32;  // block records and block maxima staged up to this many chunks per row
constexpr int kPayStage = 1024;   // payload words staged
constexpr int kKeyCap = 512;      // top-F candidate keys of a row merge
struct Stage {
  ChunkStat cs[2][kMaxChunks];         // chunk records: target row, draft row
  BlockRec blk[kStageChunks];          // block records of the row drawn from
  uint32_t bmk[kStageChunks * kBlocks];  // block maximum keys of the draft row (top-F)
  float z[2][32 * 8];                  // target / draft row values of the block a draw located
  int32_t pay[kPayStage];              // the sequence's cache payload
  uint64_t ck[kKeyCap];                // top-F candidate keys
};
static_assert(sizeof(Stage) <= kChunkBytes, "the merge stage must fit the chunk buffer");
static_assert(offsetof(Smem, hist) % 16 == 0 && offsetof(Stage, bmk) % 16 == 0 && offsetof(Stage, blk) % 16 == 0,
              "shared arrays read or copied in 16-byte pieces");
static_assert(sizeof(ChunkStat) == 16 && sizeof(BlockRec) % 16 == 0 && sizeof(RowInfo) == 32 && sizeof(PosInfo) == 16,
              "records are copied in 16-byte pieces");

// Thread 0: bounded wait (sleeping between polls) until *ctr reaches `target`,
// then an acquire; false when the wait ran out.  Used only for counts that
// CTAs which started earlier raise, so the wait ends unless they failed.
SSD_DEV bool wait_count(const uint32_t *ctr, uint32_t target) {
  for (uint32_t it = 0; it < kMaxPolls; ++it) {
    if (ld_relaxed(ctr) >= target) {
      fence_acq_rel();
      return true;
    }
    __nanosleep(200);
  }
  return false;
}

// ===========================================================================
// element access and weights
// ===========================================================================
// The 16-byte vector at chunk-local element i0 of a row chunk starting at e0
// with n elements, from global memory; elements at or past n read as `fill`.
template <class E>
SSD_DEV void ld_vec(const char *row, int e0, int n, int i0, float fill, float *f) {
  if (i0 + E::kVec <= n) {
    E::unpack(__ldg(reinterpret_cast<const uint4 *>(row + static_cast<int64_t>(e0 + i0) * E::kSize)), f);
  } else {
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) f[e] = (i0 + e < n) ? E::ld(row, e0 + i0 + e) : fill;
  }
}

// Weight functors: operator()(zt, zd, idx) -> weight >= 0 with a fixed sequence
// of correctly rounded operations, so every pass over the same elements agrees.
struct WSaguaro {  // unnormalised q'_i
  float mdk, kT, C;
  uint64_t keyF;
  bool hasS;
  SSD_DEV float operator()(float, float zd, int idx) const {
    const float e = ex2(__fmaf_rn(zd, kT, -mdk));
    return (hasS && cand_key(zd, idx) >= keyF) ? __fmul_rn(e, C) : e;
  }
};
struct WTarget {  // unnormalised p_i
  float mtk, kT;
  SSD_DEV float operator()(float zt, float, int) const { return ex2(__fmaf_rn(zt, kT, -mtk)); }
};
struct WResidual {  // max(0, p_i - q'_i)
  float mtk, kT, inv_st, mdk, fC, f1;
  uint64_t keyF;
  bool hasS;
  SSD_DEV float operator()(float zt, float zd, int idx) const {
    const float p = __fmul_rn(ex2(__fmaf_rn(zt, kT, -mtk)), inv_st);
    const float f = (hasS && cand_key(zd, idx) >= keyF) ? fC : f1;
    const float q = __fmul_rn(ex2(__fmaf_rn(zd, kT, -mdk)), f);
    const float r = __fsub_rn(p, q);
    return r > 0.f ? r : 0.f;
  }
};

// A block is the 32 consecutive vectors (256 j + 32 w + lane) warp w reads in
// round j.  Within a block the running weight has a fixed order: each lane
// sums its vector's weights in element order, the lanes are combined by a
// Hillis-Steele inclusive scan; the block's sum is the scan's last value.
SSD_DEV float warp_incl_scan(float x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = __fadd_rn(x, t);
  }
  return x;
}

// This lane's weights of its vector of block (round j, warp w) of chunk c; the
// return value is their sum in element order.
template <class E, bool HT, bool HD, class WF>
SSD_DEV float lane_weights(const VocabArgs &a, const char *rowT, const char *rowD, int c, int j, int w, const WF &wf,
                           float *x) {
  const int lane = threadIdx.x & 31;
  const int e0 = c * a.chunk_elems;
  const int n = min(a.chunk_elems, a.V - e0);
  const int i0 = (j * kThreads + w * 32 + lane) * E::kVec;
  float ft[E::kVec], fd[E::kVec];
  if constexpr (HT) ld_vec<E>(rowT, e0, n, i0, 0.f, ft);
  if constexpr (HD) ld_vec<E>(rowD, e0, n, i0, 0.f, fd);
  float p = 0.f;
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) {
    x[e] = (i0 + e < n) ? wf(HT ? ft[e] : 0.f, HD ? fd[e] : 0.f, e0 + i0 + e) : 0.f;
    p = __fadd_rn(p, x[e]);
  }
  return p;
}

// One warp: the first element of block (c, j, w) whose running weight exceeds
// `target` with positive weight; when rounding leaves the target in a lane that
// has no such element, that lane's last positive element; when no lane holds
// it, the block's last positive element; -1 for a block without weight.  All
// 32 lanes call; all return the result.  *dist (every lane) is the distance
// of the target from the nearer edge of the chosen element's bin in the
// block's running weight, 0 for the fallbacks (a near-tie by construction).
template <class E, bool HT, bool HD, class WF>
SSD_DEV int warp_find(const VocabArgs &a, const char *rowT, const char *rowD, int c, int j, int w, float target,
                      const WF &wf, float *dist) {
  const int lane = threadIdx.x & 31;
  float x[E::kVec];
  const float p = lane_weights<E, HT, HD>(a, rowT, rowD, c, j, w, wf, x);
  const float incl = warp_incl_scan(p);
  float ex = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) ex = 0.f;
  const int i0 = c * a.chunk_elems + (j * kThreads + w * 32 + lane) * E::kVec;
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
  const bool cross = p > 0.f && __fadd_rn(ex, p) > target;
  const uint32_t mc = __ballot_sync(0xffffffffu, cross);
  if (mc) {
    const int src = __ffs(mc) - 1;
    *dist = __shfl_sync(0xffffffffu, hit >= 0 ? fmaxf(edge, 0.f) : 0.f, src);
    return __shfl_sync(0xffffffffu, hit >= 0 ? hit : lpos, src);
  }
  *dist = 0.f;
  int best = lpos;
#pragma unroll
  for (int o = 16; o; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  return best;
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

// One warp: the first of n masses whose cumulative sum (warp_runs) exceeds
// the target (u * total, or u itself when u_is_target), with positive mass;
// rounding past the end takes the last positive one.  Lane 0 sets
// sh.ival[0] = its index (-1 when the total is 0), sh.scal[1] = the target
// minus the mass before it, sh.scal[2] = the total.  The caller synchronises.
SSD_DEV void locate(const float *mass, int n, float u, bool u_is_target, Smem &sh) {
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
  const uint32_t mh = __ballot_sync(0xffffffffu, hit >= 0);
  if (mh) {
    const int src = __ffs(mh) - 1;
    idx = __shfl_sync(0xffffffffu, hit, src);
    before = __shfl_sync(0xffffffffu, hb, src);
  } else {  // rounding left the target past the end: the last positive mass
    const uint32_t ml = __ballot_sync(0xffffffffu, lpos >= 0);
    if (ml) {
      const int src = 31 - __clz(ml);
      idx = __shfl_sync(0xffffffffu, lpos, src);
      before = __shfl_sync(0xffffffffu, lb, src);
    }
  }
  if (lane == 0) {
    sh.ival[0] = (W > 0.f) ? idx : -1;
    sh.scal[1] = __fsub_rn(target, before);
    sh.scal[2] = W;
  }
}

// ===========================================================================
// k_stats: statistics of one staged chunk
// ===========================================================================
// Thread t owns the chunk's vectors t + 256 j (round j); vector nvec, when the
// row's last chunk ends inside it, is read from global memory (-inf past the
// end).
template <class E>
struct ChunkView {
  const uint4 *v4;
  const char *row;
  int e0, n, nvec, ntail;
  SSD_DEV bool has(int v) const { return v < nvec || (v == nvec && ntail > 0); }
  SSD_DEV void get(int v, float *f) const {
    if (v < nvec) E::unpack(v4[v], f);
    else ld_vec<E>(row, e0, n, v * E::kVec, -__int_as_float(0x7f800000), f);
  }
  // maximum of vector v (-inf if absent)
  SSD_DEV float vmax(int v) const {
    const float NEG_INF = -__int_as_float(0x7f800000);
    if (v < nvec) {
      const uint4 w = v4[v];
      if constexpr (E::kSize == 2) {
        const uint32_t t = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
        return fmaxf(__uint_as_float(t << 16), __uint_as_float(t & 0xFFFF0000u));
      } else {
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
      }
    }
    float m = NEG_INF;
    if (has(v)) {
      float f[E::kVec];
      get(v, f);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) m = fmaxf(m, f[e]);
    }
    return m;
  }
};

// Top-F of n distinct nonzero keys by rank (the key with r larger keys goes
// to dst[r] when r < F); slots past n are set to 0.  No barrier inside.  Up to
// 64 keys: warp w ranks keys w, w + 8, ..., its lanes comparing keys l and
// l + 32 against it (two ballots); beyond, a thread per key.
SSD_DEV void rank_select(const uint64_t *keys, int n, int F, uint64_t *dst) {
  for (int i = threadIdx.x; i < F; i += kThreads)
    if (i >= n) dst[i] = 0ull;
  if (n <= 64) {
    const int lane = threadIdx.x & 31;
    const uint64_t a0 = lane < n ? keys[lane] : 0ull, a1 = lane + 32 < n ? keys[lane + 32] : 0ull;
    for (int i = threadIdx.x >> 5; i < n; i += kWarps) {
      const uint64_t k = keys[i];
      const int rank = __popc(__ballot_sync(0xffffffffu, a0 > k)) + __popc(__ballot_sync(0xffffffffu, a1 > k));
      if (lane == 0 && rank < F) dst[rank] = k;
    }
    return;
  }
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint64_t k = keys[i];
    int rank = 0;
    for (int j = 0; j < n && rank < F; ++j) rank += (keys[j] > k) ? 1 : 0;
    if (rank < F) dst[rank] = k;
  }
}

// The 8 block sums of a warp (kRounds = 8): pr[j] is this lane's part of
// round j's block.  Recursive halving: at each step a lane keeps half of its
// rounds and adds its partner's part of them (partners 16, 8, 4 lanes apart),
// then the last four lanes of a round are summed by a butterfly.  Lane l ends
// with the sum of round l / 4.
SSD_DEV float warp_round_sums(const float (&pr)[kRounds]) {
  static_assert(kRounds == 8, "three halving steps");
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

// The 8 block maximum keys of a warp: vk[j] is this lane's vector key of
// round j (0: none).  The exchange pattern of warp_round_sums with max; lane
// l ends with the maximum of round l / 4.
SSD_DEV uint32_t warp_round_umax(const uint32_t (&vk)[kRounds]) {
  const int lane = threadIdx.x & 31;
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  uint32_t q4[4], q2[2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t keep = b4 ? vk[4 + k] : vk[k], send = b4 ? vk[k] : vk[4 + k];
    q4[k] = max(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t keep = b3 ? q4[2 + k] : q4[k], send = b3 ? q4[k] : q4[2 + k];
    q2[k] = max(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  uint32_t q = max(b2 ? q2[1] : q2[0], __shfl_xor_sync(0xffffffffu, b2 ? q2[0] : q2[1], 4));
  q = max(q, __shfl_xor_sync(0xffffffffu, q, 2));
  q = max(q, __shfl_xor_sync(0xffffffffu, q, 1));
  return q;
}

// The chunk's record, block sums and (top-F rows) block maximum keys.
template <class E>
SSD_DEV void stats_chunk(const VocabArgs &a, int b, int slot, int c, const uint8_t *buf, Smem &sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowSlot rs = a.slot[slot];
  const float kT = a.kT;
  const bool greedy = a.greedy != 0;
  const float NEG_INF = -__int_as_float(0x7f800000);
  ChunkView<E> cv;
  cv.v4 = reinterpret_cast<const uint4 *>(buf);
  cv.row = row_ptr(a, rs.tensor, b, rs.row, E::kSize);
  cv.e0 = c * a.chunk_elems;
  cv.n = min(a.chunk_elems, a.V - cv.e0);
  cv.nvec = (cv.n * E::kSize) >> 4;
  cv.ntail = cv.n - cv.nvec * E::kVec;
  const bool tail_mine = cv.ntail > 0 && tid == (cv.nvec & (kThreads - 1));  // the partial vector

  // the chunk's argmax is kept where it is used: greedy rows and rows whose
  // top-1 list is the argmax (F = 1).  Elsewhere the record's index is the
  // chunk's first element, which is the argmax in the one case a T > 0 draw
  // can fall back to it (a row without finite logits: every chunk max -inf).
  const bool need_arg = greedy || rs.F == 1;
  // rows with a top-F list (F > 1) publish the maximum key of each block
  // (round, warp); the pair merge selects the row's top-F from them
  const bool topf = rs.F > 1;
  uint32_t vk[kRounds];  // topf rows: this lane's vector key of each round (0: no vector)
  float m1 = NEG_INF;
  int wi = kNone;
  if (need_arg) {
    // pass 1: the thread's maximum and the first of its vectors holding it
    int j1 = -1;
#pragma unroll
    for (int j = 0; j < kRounds; ++j) {
      const int v = tid + j * kThreads;
      vk[j] = 0u;
      if (cv.has(v)) {
        const float vm = cv.vmax(v);
        if (topf) vk[j] = f2ord(vm);
        if (vm > m1 || j1 < 0) {  // strictly larger: the first vector among equal maxima
          m1 = fmaxf(m1, vm);
          j1 = j;
        }
      }
    }
    const float wm1 = warp_max(m1);
    // the lane holding the warp maximum: its first element there
    int i1 = kNone;
    if (m1 == wm1 && j1 >= 0) {
      const int v = tid + j1 * kThreads;
      float f[E::kVec];
      cv.get(v, f);
#pragma unroll
      for (int e = E::kVec - 1; e >= 0; --e)
        if (f[e] == wm1 && v * E::kVec + e < cv.n) i1 = v * E::kVec + e;
    }
    wi = i1;
#pragma unroll
    for (int o = 16; o; o >>= 1) wi = min(wi, __shfl_xor_sync(0xffffffffu, wi, o));
  } else {
    // pass 1: the thread's maximum (bf16 rows: packed maxima of all vectors)
    if constexpr (E::kSize == 2) {
      uint32_t mm = 0xFF80FF80u;  // (-inf, -inf)
#pragma unroll
      for (int j = 0; j < kRounds; ++j) {
        const int v = tid + j * kThreads;
        vk[j] = 0u;
        if (v < cv.nvec) {
          const uint4 w = cv.v4[v];
          const uint32_t t = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
          mm = bmax2(mm, t);
          if (topf) vk[j] = f2ord(fmaxf(__uint_as_float(t << 16), __uint_as_float(t & 0xFFFF0000u)));
        }
      }
      m1 = fmaxf(__uint_as_float(mm << 16), __uint_as_float(mm & 0xFFFF0000u));
    } else {
#pragma unroll
      for (int j = 0; j < kRounds; ++j) {
        const int v = tid + j * kThreads;
        vk[j] = 0u;
        if (v < cv.nvec) {
          const float vm = cv.vmax(v);
          m1 = fmaxf(m1, vm);
          if (topf) vk[j] = f2ord(vm);
        }
      }
    }
    if (tail_mine) {
      const float vm = cv.vmax(cv.nvec);
      m1 = fmaxf(m1, vm);
      if (topf) {
#pragma unroll
        for (int j = 0; j < kRounds; ++j)
          if (j == cv.nvec / kThreads) vk[j] = f2ord(vm);
      }
    }
  }
  if (topf) {
    const uint32_t key = warp_round_umax(vk);
    if ((lane & 3) == 0) a.bmk[chunk_index(a, b, slot, c) * kBlocks + (lane >> 2) * kWarps + warp] = key;
  }
  const float wm = warp_max(m1);
  // pass 2: the warp's sum of 2^(z kT - fl(wm kT)), two elements per packed
  // FMA / ADD; per round the lane's four pairs first, then into the lane's
  // total (the same arithmetic whether or not block sums are kept).  Rows
  // that are drawn from also keep their block sums.
  float s = 0.f;
  BlockRec *br = a.blk + chunk_index(a, b, slot, c);
  if (!greedy && wm != NEG_INF) {
    const float Mk = __fmul_rn(wm, kT);
    const uint64_t k2 = pack2(kT, kT), nm2 = pack2(-Mk, -Mk);
    float tail = 0.f;  // the partial vector's sum, element order
    if (tail_mine) {
      float f[E::kVec];
      cv.get(cv.nvec, f);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) tail = __fadd_rn(tail, ex2(__fmaf_rn(f[e], kT, -Mk)));
    }
    uint64_t acc = pack2(0.f, 0.f);
    float pr[kRounds];  // block rows: the lane's sum of each round
#pragma unroll
    for (int j = 0; j < kRounds; ++j) {
      const int v = tid + j * kThreads;
      pr[j] = 0.f;
      if (v < cv.nvec) {
        const uint4 w = cv.v4[v];
        uint64_t accj = 0;
#pragma unroll
        for (int h = 0; h < E::kPairs; ++h) {
          float x0, x1;
          unpack2(fma2(E::pair(w, h), k2, nm2), x0, x1);
          const uint64_t e2 = pack2(ex2(x0), ex2(x1));
          accj = (h == 0) ? e2 : add2(accj, e2);
        }
        acc = add2(acc, accj);
        if (rs.blocks) {
          float lo, hi;
          unpack2(accj, lo, hi);
          pr[j] = __fadd_rn(lo, hi);
        }
      } else if (tail_mine && v == cv.nvec) {
        pr[j] = tail;
      }
    }
    if (rs.blocks) {
      const float bsum = warp_round_sums(pr);
      if ((lane & 3) == 0) br->bs[lane >> 2][warp] = bsum;
    }
    float lo, hi;
    unpack2(acc, lo, hi);
    s = __fadd_rn(__fadd_rn(lo, hi), tail);
    s = warp_sum(s);
  } else if (rs.blocks && lane < kRounds) {
    br->bs[lane][warp] = 0.f;  // every block record of a drawn row is written
  }
  if (lane == 0) {
    if (rs.blocks) br->wm[warp] = wm;
    sh.wm[warp] = wm;
    sh.ws[warp] = s;
    sh.wa[warp] = wi;
  }
  __syncthreads();
  if (warp == 0) {
    // lanes 0..7 hold the warps' records; reduced within groups of 8 lanes
    const int w = lane & (kWarps - 1);
    const float wmw = sh.wm[w];
    float M = wmw;
#pragma unroll
    for (int o = kWarps / 2; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    int amax = (wmw == M) ? sh.wa[w] : kNone;
#pragma unroll
    for (int o = kWarps / 2; o; o >>= 1) amax = min(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float S = 0.f;
    if (!greedy && M != NEG_INF && wmw != NEG_INF)
      S = __fmul_rn(sh.ws[w], ex2(__fsub_rn(__fmul_rn(wmw, kT), __fmul_rn(M, kT))));
#pragma unroll
    for (int o = kWarps / 2; o; o >>= 1) S = __fadd_rn(S, __shfl_xor_sync(0xffffffffu, S, o));
    if (lane == 0) {
      if (amax == kNone) amax = 0;  // an all -inf chunk: its first index
      a.stats[chunk_index(a, b, slot, c)] = ChunkStat{M, S, cv.e0 + amax, 0};
    }
  }
}

// ===========================================================================
// merges
// ===========================================================================
struct RowStat {
  float m, s;
  int amax;
};
// One warp merges the chunk records of a row (staged in shared memory): the
// maximum (a strictly larger maximum keeps the lower chunk, hence the lowest
// index), and the sum rescaled to it (each lane sums its chunks in order, the
// lanes by a fixed tree).  All 32 lanes call; all return it.
SSD_DEV RowStat merge_row_warp(const VocabArgs &a, const ChunkStat *rec) {
  constexpr int L = kMaxChunks / 32;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int lane = threadIdx.x & 31;
  ChunkStat cs[L];
#pragma unroll
  for (int l = 0; l < L; ++l) {
    const int c = lane + 32 * l;
    cs[l] = (c < a.nchunks) ? rec[c] : ChunkStat{NEG_INF, 0.f, kNone, 0};
  }
  float m = cs[0].m;
  int am = cs[0].amax;
#pragma unroll
  for (int l = 1; l < L; ++l)
    if (cs[l].m > m) {
      m = cs[l].m;
      am = cs[l].amax;
    }
  // across lanes: the larger maximum; equal maxima keep the lower index
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
    if (m2 > m || (m2 == m && a2 < am)) {
      m = m2;
      am = a2;
    }
  }
  float sum = 0.f;
  if (!a.greedy && m != NEG_INF) {
    const float mk = __fmul_rn(m, a.kT);
#pragma unroll
    for (int l = 0; l < L; ++l)
      if (cs[l].m != NEG_INF) sum = __fadd_rn(sum, __fmul_rn(cs[l].s, ex2(__fsub_rn(__fmul_rn(cs[l].m, a.kT), mk))));
    sum = warp_sum(sum);
  }
  return RowStat{m, sum, am == kNone ? 0 : am};
}

SSD_DEV float norm_N(float C, float sq) { return __fsub_rn(1.f, __fmul_rn(__fsub_rn(1.f, C), sq)); }

// ===========================================================================
// draws by the statistics of a row: chunk (chunk masses), block (block sums),
// then one warp over the block
// ===========================================================================
// Chunk masses of 2^(z kT - rk) (rk = fl(row max kT)) from the row's chunk
// records, into sh.cmass.  Caller synchronises.
SSD_DEV float chunk_mass(const ChunkStat &cs, float kT, float rk) {
  return (cs.m == -__int_as_float(0x7f800000)) ? 0.f : __fmul_rn(cs.s, ex2(__fsub_rn(__fmul_rn(cs.m, kT), rk)));
}
SSD_DEV void chunk_masses(const VocabArgs &a, int b, int slot, float rk, Smem &sh) {
  for (int c = threadIdx.x; c < a.nchunks; c += kThreads)
    sh.cmass[c] = chunk_mass(ldcg_stat(a.stats + chunk_index(a, b, slot, c)), a.kT, rk);
}

// Draw from row `slot` of sequence b (its elements in `row`) with weights wf =
// 2^(z kT - rk), scaled by C on the set S (the Fn keys of Slist) when C < 1.
// sh.cmass holds the chunk masses with the down-weighting applied; `sbr`, when
// given, the row's block records staged in shared memory (else they are read
// from global memory).  While warp 0 scans the located block, warp 1 stages
// its values (zdrawn) and, with `rowZ`, the other row's values there
// (zother); sh.ival[5] is then the block's first element.  Every thread
// calls; returns the token (-1 if the masses are all 0).
template <class E, bool HT, class WF>
SSD_DEV int stats_draw(const VocabArgs &a, int b, int slot, const char *row, float rk, float u, const WF &wf,
                       const BlockRec *sbr, const uint64_t *Slist, int Fn, float C, float *zdrawn, const char *rowZ,
                       float *zother, Smem &sh) {
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) sh.near = 0;
  if (warp == 0) locate(sh.cmass, a.nchunks, u, false, sh);
  __syncthreads();
  const int cs = sh.ival[0];
  const float local = sh.scal[1];
  const float Wrow = sh.scal[2];  // the row's total weight
  if (cs < 0) return -1;
  // block weights of chunk cs; the elements of S in a block down-weighted in
  // list order
  if (tid < kBlocks) {
    const int j = tid / kWarps, w = tid % kWarps;
    float wmw, bs;
    if (sbr) {
      wmw = sbr[cs].wm[w];
      bs = sbr[cs].bs[j][w];
    } else {
      const BlockRec *br = a.blk + chunk_index(a, b, slot, cs);
      wmw = __ldcg(&br->wm[w]);
      bs = __ldcg(&br->bs[j][w]);
    }
    float x = (wmw == -__int_as_float(0x7f800000) || !(bs > 0.f))
                  ? 0.f
                  : __fmul_rn(bs, ex2(__fsub_rn(__fmul_rn(wmw, a.kT), rk)));
    if (C < 1.f) {
      const int e0 = cs * a.chunk_elems;
      for (int i = 0; i < Fn; ++i) {
        const uint64_t k = Slist[i];
        if (!k) continue;
        const int idx = cand_idx(k) - e0;
        if (idx < 0 || idx >= a.chunk_elems) continue;
        const int v = idx / E::kVec;
        if ((v / kThreads) * kWarps + (v % kThreads) / 32 != tid) continue;
        const float e = ex2(__fmaf_rn(cand_val(k), a.kT, -rk));
        x = fmaxf(__fsub_rn(x, __fmul_rn(__fsub_rn(1.f, C), e)), 0.f);
      }
    }
    sh.bw[tid] = x;
  }
  __syncthreads();
  if (warp == 0) {
    locate(sh.bw, kBlocks, local, true, sh);
    __syncwarp();
    if (tid == 0 && sh.ival[0] < 0) {  // no block weight (the masses rounded differently): the last block
      sh.ival[0] = kBlocks - 1;
      sh.scal[1] = local;
      sh.near = 1;
    }
  }
  __syncthreads();
  const int blk = sh.ival[0];
  const float local2 = sh.scal[1];
  int d = -1;
  float dist = 0.f;
  if (warp == 0) {
    d = warp_find<E, HT, !HT>(a, HT ? row : nullptr, HT ? nullptr : row, cs, blk / kWarps, blk % kWarps, local2,
                              wf, &dist);
  } else if (warp == 1 && zdrawn) {
    const int lane = tid & 31;
    const int e0 = cs * a.chunk_elems;
    const int n = min(a.chunk_elems, a.V - e0);
    const int i0 = ((blk / kWarps) * kThreads + (blk % kWarps) * 32 + lane) * E::kVec;
    float f[E::kVec], g[E::kVec];
    ld_vec<E>(row, e0, n, i0, 0.f, f);
    if (rowZ) ld_vec<E>(rowZ, e0, n, i0, 0.f, g);
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) zdrawn[lane * E::kVec + e] = f[e];
    if (rowZ)
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) zother[lane * E::kVec + e] = g[e];
  }
  __syncthreads();  // everyone read sh.ival / sh.scal
  if (tid == 0) {
    sh.ival[4] = d;
    sh.ival[5] = cs * a.chunk_elems + ((blk / kWarps) * kThreads + (blk % kWarps) * 32) * E::kVec;  // zbuf[0]
    if (!(dist >= __fmul_rn(kNearTie, Wrow))) sh.near = 1;
  }
  __syncthreads();
  return sh.ival[4];
}

// A draw from a row without usable block sums (rows whose statistics kept
// none, or Saguaro weights whose down-weighting makes the statistics' masses
// inexact): exact block sums by one warp per block (the arithmetic of
// warp_find), chunk masses from them, then the located chunk's block sums
// again and one warp over the located block.  Every thread calls; returns the
// token (-1 when the row has no weight).
template <class E, bool HT, bool HD, class WF>
SSD_DEV int exact_draw(const VocabArgs &a, const char *rowT, const char *rowD, float u, const WF &wf, Smem &sh) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto block_sums = [&](int c) {  // sh.bw[0..kBlocks) of chunk c
    for (int k = warp; k < kBlocks; k += kWarps) {
      float x[E::kVec];
      const float p = lane_weights<E, HT, HD>(a, rowT, rowD, c, k / kWarps, k % kWarps, wf, x);
      const float incl = warp_incl_scan(p);
      if (lane == 31) sh.bw[k] = incl;
    }
    __syncthreads();
  };
  for (int c = 0; c < a.nchunks; ++c) {
    block_sums(c);
    if (warp == 0) {
      const float m = warp_total(sh.bw, kBlocks);
      if (lane == 0) sh.cmass[c] = m;
    }
    __syncthreads();
  }
  if (tid == 0) sh.near = 0;
  if (warp == 0) locate(sh.cmass, a.nchunks, u, false, sh);
  __syncthreads();
  const int cs = sh.ival[0];
  const float local = sh.scal[1];
  const float Wrow = sh.scal[2];  // the row's total weight
  if (cs < 0) return -1;
  __syncthreads();
  block_sums(cs);
  if (warp == 0) locate(sh.bw, kBlocks, local, true, sh);
  __syncthreads();
  const int blk = sh.ival[0];
  const float local2 = sh.scal[1];
  int d = -1;
  float dist = 0.f;
  if (warp == 0 && blk >= 0)
    d = warp_find<E, HT, HD>(a, rowT, rowD, cs, blk / kWarps, blk % kWarps, local2, wf, &dist);
  __syncthreads();
  if (tid == 0) {
    sh.ival[4] = d;
    if (!(dist >= __fmul_rn(kNearTie, Wrow))) sh.near = 1;
  }
  __syncthreads();
  return sh.ival[4];
}

// p_{r+1} (target row r) drawn by its statistics; the row's argmax if the
// masses are all zero.  `st`: the row's chunk (and, up to kStageChunks
// chunks, block) records staged by stage_chain (target row K only).
template <class E>
SSD_DEV int draw_target(const VocabArgs &a, int b, int r, const RowInfo &row, float u, const Stage *st, Smem &sh) {
  const float mtk = __fmul_rn(row.mt, a.kT);
  const WTarget wp{mtk, a.kT};
  const char *rowT = row_ptr(a, 0, b, r, E::kSize);
  int d;
  if (a.slot[a.tsl[r]].blocks) {
    const BlockRec *sbr = nullptr;
    if (st) {
      for (int c = threadIdx.x; c < a.nchunks; c += kThreads) sh.cmass[c] = chunk_mass(st->cs[0][c], a.kT, mtk);
      if (a.nchunks <= kStageChunks) sbr = st->blk;
    } else {
      chunk_masses(a, b, a.tsl[r], mtk, sh);
    }
    __syncthreads();
    d = stats_draw<E, true>(a, b, a.tsl[r], rowT, mtk, u, wp, sbr, nullptr, 0, 1.f, nullptr, nullptr, nullptr, sh);
  } else {
    d = exact_draw<E, true, false>(a, rowT, nullptr, u, wp, sh);
  }
  return (d >= 0) ? d : row.at;
}

SSD_DEV WResidual residual_weights(const VocabArgs &a, const RowInfo &ri, uint64_t keyF, int F) {
  WResidual wf;
  wf.mtk = __fmul_rn(ri.mt, a.kT);
  wf.kT = a.kT;
  wf.inv_st = __frcp_rn(ri.st);
  wf.mdk = __fmul_rn(ri.md, a.kT);
  const float sN = __fmul_rn(ri.sd, norm_N(a.C, ri.sq));
  wf.f1 = __frcp_rn(sN);
  wf.fC = __fdiv_rn(a.C, sN);
  wf.hasS = F > 0;
  wf.keyF = keyF;
  return wf;
}

// ===========================================================================
// the row's top-F from its block maximum keys
// ===========================================================================
// The elements (value descending, index ascending) of block `blk` (chunk
// blk / kBlocks, round, warp) that this lane reads: its 16-byte vector.
template <class E>
SSD_DEV void block_vec(const VocabArgs &a, const char *row, int blk, float *f, int *i0, int *n) {
  const int lane = threadIdx.x & 31;
  const int c = blk / kBlocks, k = blk - c * kBlocks;
  const int e0 = c * a.chunk_elems;
  *n = min(a.chunk_elems, a.V - e0) + e0;
  *i0 = e0 + ((k / kWarps) * kThreads + (k % kWarps) * 32 + lane) * E::kVec;
  ld_vec<E>(row, e0, *n - e0, *i0 - e0, -__int_as_float(0x7f800000), f);
}

// The top-F (F > 1) of a draft row into sh.S (descending; zeros past the
// row's elements).  t16 = the 16-bit key prefix of the F-th largest block
// maximum (two levels of 256-bucket counts): at least F elements reach it,
// so the row's top-F all lie in blocks whose maximum does.  Those blocks are
// read again (one warp per block) and their elements reaching t16 ranked;
// when ties overflow the buffers, F sweeps of a CTA-wide maximum instead.
// sh.hist, sh.ncand and sh.ival[7] start at zero.  Every thread calls.
template <class E>
SSD_DEV void row_topf(const VocabArgs &a, const char *row, int F, const uint32_t *bmk, bool staged, Stage &st,
                      Smem &sh) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nb = a.nchunks * kBlocks;
  const int lane = tid & 31;
  auto key_at = [&](int i) -> uint32_t { return staged ? bmk[i] : __ldcg(bmk + i); };
  // Bucket counts, one add per distinct bucket of a warp's 32 keys (block
  // maxima of one row crowd into a few buckets; adding key by key would
  // serialise the shared-memory atomics on them).  The loops run whole warps.
  auto count = [&](uint32_t *hist, bool v, uint32_t bucket) {
    const uint32_t peers = __match_any_sync(0xffffffffu, v ? bucket : 0xFFFFFFFFu);
    if (v && lane == __ffs(peers) - 1) atomicAdd(&hist[bucket], static_cast<uint32_t>(__popc(peers)));
  };
  for (int i0 = warp * 32; i0 < nb; i0 += kThreads) {
    const uint32_t k = (i0 + lane < nb) ? key_at(i0 + lane) : 0u;
    count(sh.hist[0], k != 0u, k >> 24);
  }
  __syncthreads();
  uint32_t b1, b2;
  int above, above2;
  find_bucket(sh.hist[0], F, b1, above);
  for (int i0 = warp * 32; i0 < nb; i0 += kThreads) {
    const uint32_t k = (i0 + lane < nb) ? key_at(i0 + lane) : 0u;
    count(sh.hist[1], k != 0u && (k >> 24) == b1, (k >> 16) & 0xFFu);
  }
  __syncthreads();
  find_bucket(sh.hist[1], F - above, b2, above2);
  const uint32_t t16 = (b1 << 8) | b2;
  // the candidate blocks
  constexpr int kListCap = kCandCap * 2;
  int *blist = reinterpret_cast<int *>(sh.cand);
  for (int i = tid; i < nb; i += kThreads) {
    const uint32_t k = key_at(i);
    if (k && (k >> 16) >= t16) {
      const int p = atomicAdd(&sh.ival[7], 1);
      if (p < kListCap) blist[p] = i;
    }
  }
  __syncthreads();
  const int nbl = sh.ival[7];
  const bool listed = nbl <= kListCap;
  if (listed) {
    for (int q = warp; q < nbl; q += kWarps) {
      float f[E::kVec];
      int i0, n;
      block_vec<E>(a, row, blist[q], f, &i0, &n);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e)
        if (i0 + e < n && (f2ord(f[e]) >> 16) >= t16) {
          const int p = atomicAdd(&sh.ncand, 1);
          if (p < kKeyCap) st.ck[p] = cand_key(f[e], i0 + e);
        }
    }
  }
  __syncthreads();
  const int nc = sh.ncand;
  if (listed && nc <= kKeyCap) {
    rank_select(st.ck, nc, F, sh.S);
  } else {
    // ties at the threshold: one winner per sweep over the candidate blocks
    // (every block when they overflow the list)
    const int nq = listed ? nbl : nb;
    uint64_t prev = ~0ull;
    for (int r = 0; r < F; ++r) {
      uint64_t best = 0ull;
      for (int q = warp; q < nq; q += kWarps) {
        float f[E::kVec];
        int i0, n;
        block_vec<E>(a, row, listed ? blist[q] : q, f, &i0, &n);
#pragma unroll
        for (int e = 0; e < E::kVec; ++e) {
          if (i0 + e >= n || (f2ord(f[e]) >> 16) < t16) continue;
          const uint64_t key = cand_key(f[e], i0 + e);
          if (key < prev && key > best) best = key;
        }
      }
      best = block_max_u64<kThreads>(best, sh.redk);
      if (tid == 0) sh.S[r] = best;
      prev = best;
    }
  }
  __syncthreads();
}

// ===========================================================================
// pair merge: row statistics, top-F list, Saguaro draw, p(d), q'(d), guesses
// ===========================================================================
template <class E>
__device__ __forceinline__ void row_finish(const VocabArgs &a, int b, int r, Stage &st, Smem &sh) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ts = a.tsl[r], ds = a.dsl[r];
  const int F = (ds >= 0) ? a.Fs[r] : 0;
  const size_t rr = static_cast<size_t>(b) * (a.K + 1) + r;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const char *rowT = row_ptr(a, 0, b, r, E::kSize);
  const char *rowD = row_ptr(a, 1, b, r, E::kSize);
  const bool draws = r < a.K && a.do_sample && !a.greedy && ds >= 0;
  const bool stage_blk = draws && a.slot[ds].blocks && a.nchunks <= kStageChunks;
  const bool given = r < a.K && !a.do_sample && a.do_verify;  // verification of tokens the caller drew
  const bool stage_bmk = F > 1 && a.nchunks <= kStageChunks;
  // one round of loads: both rows' chunk records, the draft row's block
  // maximum keys (top-F), the block records of a row drawn from and (tokens
  // given) the token with its two logits
  const uint32_t *gbmk = a.bmk + chunk_index(a, b, ds, 0) * kBlocks;
  if (stage_bmk)
    for (int i = tid; i < a.nchunks * (kBlocks / 4); i += kThreads)
      cp_async16(reinterpret_cast<int4 *>(st.bmk) + i, reinterpret_cast<const int4 *>(gbmk) + i);
  if (F > 1) {
    sh.hist[0][tid] = 0u;
    sh.hist[1][tid] = 0u;
  }
  for (int c = tid; c < a.nchunks; c += kThreads) {
    if (ts >= 0) cp_async16(&st.cs[0][c], a.stats + chunk_index(a, b, ts, c));
    if (ds >= 0) cp_async16(&st.cs[1][c], a.stats + chunk_index(a, b, ds, c));
  }
  if (stage_blk) {
    constexpr int kW = static_cast<int>(sizeof(BlockRec) / 16);
    const int4 *src = reinterpret_cast<const int4 *>(a.blk + chunk_index(a, b, ds, 0));
    int4 *dst = reinterpret_cast<int4 *>(st.blk);
    for (int i = tid; i < a.nchunks * kW; i += kThreads) cp_async16(dst + i, src + i);
  }
  if (tid == 0) {
    memset(&sh.ri, 0, sizeof(sh.ri));
    sh.ncand = 0;
    sh.ival[7] = 0;
    if (given) {
      const int d = a.d_in[static_cast<size_t>(b) * a.K + r];
      sh.ival[2] = d;
      if (d >= 0 && d < a.V && !a.greedy) {
        sh.scal[4] = E::ld(rowT, d);
        sh.scal[5] = E::ld(rowD, d);
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();
  // the last two warps merge the target and draft rows' chunk records; all
  // warps then select the draft row's top-F
  if (warp == kWarps - 2 && ts >= 0) {
    const RowStat t = merge_row_warp(a, st.cs[0]);
    if (lane == 0) {
      sh.ri.mt = t.m;
      sh.ri.st = t.s;
      sh.ri.at = t.amax;
    }
  }
  if (warp == kWarps - 1 && ds >= 0) {
    const RowStat d = merge_row_warp(a, st.cs[1]);
    if (lane == 0) {
      sh.ri.md = d.m;
      sh.ri.sd = d.s;
      sh.ri.ad = d.amax;
    }
  }
  // the draft row's top-F list: S (and its global copy), Σ_S q and the
  // guesses of depth r
  auto list_part = [&]() {
    if (F > 1) row_topf<E>(a, rowD, F, stage_bmk ? st.bmk : gbmk, stage_bmk, st, sh);
    __syncthreads();  // the merged statistics and the list
    const float mdk = __fmul_rn(sh.ri.md, a.kT);
    if (F == 1 && tid == 0) sh.S[0] = cand_key(sh.ri.md, sh.ri.ad);  // the top-1: the row's argmax
    if (F == 1) __syncthreads();
    if (a.do_verify || a.do_lookup || a.do_analytics)
      for (int i = tid; i < F; i += kThreads) a.S[rr * a.Fcap + i] = sh.S[i];
    // the draft's normalised mass on S: lane-strided partial sums, a fixed tree
    if (warp == 0) {
      float sq = 0.f;
      if (!a.greedy && sh.ri.md != NEG_INF) {
        for (int i = lane; i < F; i += 32)
          if (sh.S[i]) sq = __fadd_rn(sq, ex2(__fmaf_rn(cand_val(sh.S[i]), a.kT, -mdk)));
        sq = __fdiv_rn(warp_sum(sq), sh.ri.sd);
      }
      if (lane == 0) sh.ri.sq = sq;
    }
    __syncthreads();
    if (a.do_predict && ds >= 0) {
      const int sumF = a.foff[a.K + 1];
      for (int i = tid; i < a.F[r]; i += kThreads) {
        const uint64_t key = sh.S[i];
        a.guess[static_cast<size_t>(b) * sumF + a.foff[r] + i] = cand_idx(key);
        if (a.guess_q) {
          float q;
          if (a.greedy) q = (i == 0) ? 1.f : 0.f;
          else q = __fdiv_rn(ex2(__fmaf_rn(cand_val(key), a.kT, -mdk)), sh.ri.sd);
          a.guess_q[static_cast<size_t>(b) * sumF + a.foff[r] + i] = q;
        }
      }
    }
  };
  // with C = 1 the draw, p(d), q'(d) and the residual weights do not depend
  // on S: the list comes after the position's verdict, which may start the
  // residual draw sooner
  const bool verdict = a.do_verify && !a.greedy && r < a.K;
  const bool late_list = verdict && !(a.C < 1.f);
  if (late_list) __syncthreads();  // the merged statistics
  else list_part();
  const float mdk = __fmul_rn(sh.ri.md, a.kT);
  const RowInfo ri = sh.ri;  // late_list: sq = 0 until the list is done (C = 1 makes q' not depend on it)
  const uint64_t keyF = (F > 0 && !late_list) ? sh.S[F - 1] : 0ull;
  mark(a, sh.mk, 3);
  if (r < a.K && (a.do_sample || a.do_verify)) {
    int d;
    bool zknown = false;  // zt / zd hold the token's logits
    float zt = 0.f, zd = 0.f;
    if (a.do_sample) {
      float qd;
      if (a.greedy) {
        d = ri.ad;
        qd = 1.f;
      } else {
        const WSaguaro wf{mdk, a.kT, a.C, keyF, F > 0};
        const float u = a.u_draft[static_cast<size_t>(b) * a.K + r];
        if (__fmul_rn(__fsub_rn(1.f, a.C), ri.sq) > 0.875f || !a.slot[ds].blocks) {
          d = exact_draw<E, false, true>(a, nullptr, rowD, u, wf, sh);
        } else {
          // chunk masses of q' (unnormalised): s_c 2^(Mk_c - mdk) - (1 - C) sum_{i in S, in c} e_i,
          // the elements of S in list order
          for (int c = tid; c < a.nchunks; c += kThreads) {
            float m = chunk_mass(st.cs[1][c], a.kT, mdk);
            if (a.C < 1.f) {
              for (int i = 0; i < F; ++i) {
                const uint64_t k = sh.S[i];
                if (!k || cand_idx(k) / a.chunk_elems != c) continue;
                m = __fsub_rn(m, __fmul_rn(__fsub_rn(1.f, a.C), ex2(__fmaf_rn(cand_val(k), a.kT, -mdk))));
              }
              m = fmaxf(m, 0.f);
            }
            sh.cmass[c] = m;
          }
          __syncthreads();
          d = stats_draw<E, false>(a, b, ds, rowD, mdk, u, wf, stage_blk ? st.blk : nullptr, sh.S, F, a.C, st.z[1],
                                   a.do_verify ? rowT : nullptr, st.z[0], sh);
          if (d >= 0) {
            const int o = d - sh.ival[5];
            if (o >= 0 && o < 32 * E::kVec) {
              zd = st.z[1][o];
              zt = st.z[0][o];
              zknown = true;
            }
          }
        }
        if (tid == 0 && sh.near && a.near_ties) atomicAdd(a.near_ties, 1u);
        if (d < 0) d = ri.ad;
        if (!zknown) {
          zd = E::ld(rowD, d);
          zt = a.do_verify ? E::ld(rowT, d) : 0.f;
          zknown = true;
        }
        const bool ins = F > 0 && cand_key(zd, d) >= keyF;
        const float q = __fdiv_rn(ex2(__fmaf_rn(zd, a.kT, -mdk)), ri.sd);
        qd = __fdiv_rn(ins ? __fmul_rn(q, a.C) : q, norm_N(a.C, ri.sq));
      }
      if (tid == 0) {
        a.d_out[static_cast<size_t>(b) * a.K + r] = d;
        if (a.qd_out) a.qd_out[static_cast<size_t>(b) * a.K + r] = qd;
      }
    } else {
      d = sh.ival[2];
      zt = sh.scal[4];
      zd = sh.scal[5];
      zknown = true;
    }
    if (a.do_verify && tid == 0) {
      PosInfo pi{d, 0.f, 0.f, 0};
      if (d >= 0 && d < a.V) {
        if (a.greedy) {
          pi.p = (d == ri.at) ? 1.f : 0.f;
          pi.q = (d == ri.ad) ? 1.f : 0.f;
        } else {
          if (!zknown) {
            zt = E::ld(rowT, d);
            zd = E::ld(rowD, d);
          }
          const bool ins = F > 0 && cand_key(zd, d) >= keyF;
          pi.p = __fdiv_rn(ex2(__fmaf_rn(zt, a.kT, -__fmul_rn(ri.mt, a.kT))), ri.st);
          const float q = __fdiv_rn(ex2(__fmaf_rn(zd, a.kT, -mdk)), ri.sd);
          pi.q = __fdiv_rn(ins ? __fmul_rn(q, a.C) : q, norm_N(a.C, ri.sq));
        }
      } else {
        pi.p = -1.f;
        atomicOr(a.status, kFlagBadToken);
      }
      a.pos[static_cast<size_t>(b) * a.K + r] = pi;
      if (a.accept_prob) {
        float ap;
        if (pi.p < 0.f) ap = 0.f;
        else if (pi.q > 0.f) ap = fminf(1.f, __fdiv_rn(pi.p, pi.q));
        else ap = (pi.p > 0.f) ? 1.f : 0.f;
        a.accept_prob[static_cast<size_t>(b) * a.K + r] = ap;
      }
    }
  }
  if (tid == 0) a.rows[rr] = ri;
  if (verdict) {
    // the position's verdict (1 accepted, 2 rejected; + 2 once the pair's
    // list is also written), then the frontier: once the positions before the
    // first rejection are all accepted, the residual draw may start (ready
    // word = rejected position + 2) without waiting for the remaining pairs
    __syncthreads();  // the pair's results are written
    uint32_t vword = 0;
    if (tid == 0) {
      const PosInfo pi = ldcg_pos(a.pos + static_cast<size_t>(b) * a.K + r);
      const bool ok = pi.p >= 0.f && __fmul_rn(a.u_acc[static_cast<size_t>(b) * a.K + r], pi.q) < pi.p;
      vword = (ok ? 1u : 2u) + (late_list ? 0u : 2u);
      st_release(pos_verdict(a, b, r), vword);
      uint32_t v[kMaxK];  // every verdict load in flight at once
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) v[j] = (j < a.K) ? ld_relaxed(pos_verdict(a, b, j)) : 1u;
      uint32_t acc_mask = 0, rej_mask = 0;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (v[j] == 1u || v[j] == 3u) acc_mask |= 1u << j;
        if (v[j] == 2u || v[j] == 4u) rej_mask |= 1u << j;
      }
      const uint32_t open = ~acc_mask;  // the first position not known to be accepted
      if (open) {
        const int j = __ffs(static_cast<int>(open)) - 1;
        if ((rej_mask >> j) & 1u) {
          fence_acq_rel();  // the verdicts (and results) of positions 0..j, then the ready word
          atomicCAS(ready_word(a, b), 0u, static_cast<uint32_t>(j + 2));
        }
      }
    }
    if (late_list) {
      list_part();
      if (tid == 0) a.rows[rr] = sh.ri;  // with Σ_S q
      __syncthreads();                   // the list is written
      if (tid == 0) st_release(pos_verdict(a, b, r), vword + 2u);
    }
  }
}

// ===========================================================================
// sequence finish: acceptance chain, bonus draw, outputs, cache lookup
// ===========================================================================
// The top-F lists of a sequence (cache lookup) fit sh.cand; its payload fits
// the payload stage.
SSD_DEV bool lists_staged(const VocabArgs &a) { return a.do_lookup && a.foff[a.K + 1] <= kCandCap; }
SSD_DEV bool pay_staged(const VocabArgs &a) {
  return a.do_lookup && a.next_tokens && a.payload && a.foff[a.K + 1] * a.K <= kPayStage;
}

// Stage in shared memory, in one round of loads, what the final steps of
// sequence b need whatever the accept count: draft tokens, p(d), q'(d), the
// uniforms, every row's merged statistics and S threshold key, the top-F
// lists (sh.cand) and payload (`pay`) of the cache lookup when they fit, the
// residual unit masses (`umass`) and target row K's chunk and block records
// for the bonus draw (`st`).  Then the acceptance chain (thread 0).  Every
// thread returns the accept count.
SSD_DEV void stage_issue(const VocabArgs &a, int b, int32_t *pay, Stage *st, bool lists, Smem &sh);
SSD_DEV void stage_lists(const VocabArgs &a, int b, Smem &sh);
SSD_DEV int stage_complete(const VocabArgs &a, Smem &sh);
SSD_DEV int stage_chain(const VocabArgs &a, int b, float *umass, int32_t *pay, Stage *st, Smem &sh) {
  stage_issue(a, b, pay, st, true, sh);
  if (umass) {
    const int nu = a.nchunks * kQuarters;
    for (int q = threadIdx.x; q < nu; q += kThreads) cp_async4(&umass[q], a.rmass + static_cast<size_t>(b) * nu + q);
  }
  return stage_complete(a, sh);
}
// The top-F lists of the cache lookup (when they fit sh.cand), issued
// (cp.async) without a wait.
SSD_DEV void stage_lists(const VocabArgs &a, int b, Smem &sh) {
  if (!lists_staged(a)) return;
  const size_t r0 = static_cast<size_t>(b) * (a.K + 1);
  const int nS = a.foff[a.K + 1];
  for (int i = threadIdx.x; i < nS; i += kThreads) {
    int r = 0;
    while (i >= a.foff[r + 1]) ++r;
    cp_async8(&sh.cand[i], a.S + (r0 + r) * a.Fcap + (i - a.foff[r]));
  }
}
// The loads of stage_chain but the unit masses (and, unless `lists`, the
// lookup lists), issued (cp.async) without a wait.
SSD_DEV void stage_issue(const VocabArgs &a, int b, int32_t *pay, Stage *st, bool lists, Smem &sh) {
  const int tid = threadIdx.x;
  const size_t r0 = static_cast<size_t>(b) * (a.K + 1);
  for (int t = tid; t < a.K; t += kThreads) {
    cp_async16(&sh.pos[t], a.pos + static_cast<size_t>(b) * a.K + t);
    cp_async4(&sh.cu[t], a.u_acc + static_cast<size_t>(b) * a.K + t);
  }
  for (int i = tid; i < 2 * (a.K + 1); i += kThreads)
    cp_async16(reinterpret_cast<int4 *>(&sh.rows[i >> 1]) + (i & 1), reinterpret_cast<const int4 *>(a.rows + r0 + (i >> 1)) + (i & 1));
  for (int r = tid; r <= a.K; r += kThreads) {
    const int F = a.Fs[r];
    if (F > 0) cp_async8(&sh.keyF[r], a.S + (r0 + r) * a.Fcap + F - 1);
    else sh.keyF[r] = 0ull;
  }
  if (lists) stage_lists(a, b, sh);
  if (pay && pay_staged(a)) {
    const int n = a.foff[a.K + 1] * a.K;
    const int32_t *src = a.payload + static_cast<size_t>(b) * n;
    for (int i = tid; i < n; i += kThreads) cp_async4(&pay[i], src + i);
  }
  if (st && !a.greedy && a.tsl[a.K] >= 0) {
    const int ts = a.tsl[a.K];
    for (int c = tid; c < a.nchunks; c += kThreads) cp_async16(&st->cs[0][c], a.stats + chunk_index(a, b, ts, c));
    if (a.slot[ts].blocks && a.nchunks <= kStageChunks) {
      constexpr int kW = static_cast<int>(sizeof(BlockRec) / 16);
      const int4 *src = reinterpret_cast<const int4 *>(a.blk + chunk_index(a, b, ts, 0));
      int4 *dst = reinterpret_cast<int4 *>(st->blk);
      for (int i = tid; i < a.nchunks * kW; i += kThreads) cp_async16(dst + i, src + i);
    }
  }
}
// Waits for the staged loads, then the acceptance chain; every thread returns
// the accept count.
SSD_DEV int stage_complete(const VocabArgs &a, Smem &sh) {
  const int tid = threadIdx.x;
  cp_async_wait_all();
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int t = 0; t < a.K; ++t) {
      const PosInfo pi = sh.pos[t];
      if (pi.p >= 0.f && __fmul_rn(sh.cu[t], pi.q) < pi.p) ++acc;
      else break;
    }
    sh.ival[1] = acc;
  }
  __syncthreads();
  return sh.ival[1];
}

// Outputs of sequence b once its bonus token bt is known (sh.cd: draft tokens;
// the lookup's lists and payload as stage_chain staged them, `pay` its
// payload stage).
SSD_DEV void emit(const VocabArgs &a, int b, int acc, int bt, float W, bool zero, bool near_bonus, const int32_t *pay,
                  Smem &sh) {
  const int tid = threadIdx.x;
  const int Fa = a.F[acc];
  if (tid == 0) {
    sh.ival[3] = kNone;
    if (a.near_ties && !a.greedy) {
      // the acceptance tests actually taken (positions 1..acc+1) whose u lies
      // within kNearTie of p/q', and the bonus draw
      uint32_t n = near_bonus ? 1u : 0u;
      for (int t = 0; t <= acc && t < a.K; ++t) {
        const PosInfo pi = sh.pos[t];
        if (pi.p >= 0.f && pi.q > 0.f && fabsf(__fsub_rn(sh.cu[t], __fdiv_rn(pi.p, pi.q))) < kNearTie) ++n;
      }
      if (n) atomicAdd(a.near_ties, n);
    }
  }
  __syncthreads();
  if (a.do_lookup) {
    if (lists_staged(a)) {
      for (int i = tid; i < Fa; i += kThreads)
        if (cand_idx(sh.cand[a.foff[acc] + i]) == bt) atomicMin(&sh.ival[3], i);
    } else {
      const uint64_t *S = a.S + (static_cast<size_t>(b) * (a.K + 1) + acc) * a.Fcap;
      for (int i = tid; i < Fa; i += kThreads)
        if (cand_idx(ldcg_key(S + i)) == bt) atomicMin(&sh.ival[3], i);
    }
    __syncthreads();
  }
  const int s_hit = (a.do_lookup && sh.ival[3] != kNone) ? a.foff[acc] + sh.ival[3] : -1;
  if (tid <= a.K) {
    int v = -1;
    if (tid < acc) v = sh.pos[tid].d;
    if (tid == acc) v = bt;
    a.out_tokens[static_cast<size_t>(b) * (a.K + 1) + tid] = v;
  }
  if (a.do_lookup && a.next_tokens && tid < a.K) {
    int v = -1;
    if (s_hit >= 0 && a.payload)
      v = (pay && pay_staged(a)) ? pay[s_hit * a.K + tid]
                                 : a.payload[(static_cast<size_t>(b) * a.foff[a.K + 1] + s_hit) * a.K + tid];
    a.next_tokens[static_cast<size_t>(b) * a.K + tid] = v;
  }
  __syncthreads();
  if (tid == 0) {
    if (zero) atomicOr(a.status, kFlagZeroResidual);
    a.accept_len[b] = acc;
    a.bonus[b] = bt;
    if (a.resid_mass) a.resid_mass[b] = W;
    if (a.do_lookup) {
      if (a.slot_out) a.slot_out[b] = s_hit;
      if (s_hit >= 0) atomicAdd(a.ctr + 1, 1u);
    }
    const uint32_t done = atom_add_release(a.ctr, 1u);
    if (done + 1 == static_cast<uint32_t>(a.B) && a.hits) {
      fence_acq_rel();
      *a.hits = ld_relaxed(a.ctr + 1);
    }
  }
  __syncthreads();
}

// The last pair of sequence b merged: chain, then (greedy, or every token
// accepted) the bonus draw and the outputs; a residual draw is left to k_resid.
template <class E>
__device__ __forceinline__ void seq_finish(const VocabArgs &a, int b, Stage &st, Smem &sh) {
  const int acc = stage_chain(a, b, nullptr, st.pay, &st, sh);
  const bool resid = !a.greedy && acc < a.K;
  if (threadIdx.x == 0) {
    // the sequence's k_resid CTAs may go on (unless a pair merge's frontier
    // already set the word: to the same value); the word carries the accept
    // count + 2 (1: no residual draw)
    fence_acq_rel();
    atomicCAS(ready_word(a, b), 0u, static_cast<uint32_t>((resid ? acc : -1) + 2));
  }
  if (resid) return;
  const RowInfo row = sh.rows[acc];
  int bt = row.at;
  float W = 1.f;
  bool zero = false, near = false;
  if (a.greedy) {
    if (acc < a.K) {
      W = (row.at != row.ad) ? 1.f : 0.f;
      zero = !(W > 0.f);
    }
  } else {
    bt = draw_target<E>(a, b, acc, row, a.u_bonus[b], acc == a.K ? &st : nullptr, sh);
    near = threadIdx.x == 0 && sh.near;
  }
  emit(a, b, acc, bt, W, zero, near, st.pay, sh);
}

// The CTA's trace entry: (SM << 48 | kind << 40 | sequence << 20 | index),
// then its seven marks (0 = not reached).
SSD_DEV void trace_entry(unsigned long long *tr, int kind, int b, int idx, const unsigned long long *mk) {
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  tr[0] = (static_cast<unsigned long long>(smid) << 48) | (static_cast<unsigned long long>(kind) << 40) |
          (static_cast<unsigned long long>(b & 0xFFFFF) << 20) | static_cast<unsigned long long>(idx & 0xFFFFF);
#pragma unroll
  for (int k = 0; k < 7; ++k) tr[1 + k] = mk[k];
}

// ===========================================================================
// the kernels
// ===========================================================================
template <class E>
__global__ void __launch_bounds__(kThreads, kStatsCtas) k_stats(const __grid_constant__ VocabArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *buf = smem_raw;
  Smem &sh = *reinterpret_cast<Smem *>(smem_raw + kChunkBytes);
  // k_resid (if any) may start launching once every CTA of this grid has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  const int c = static_cast<int>(blockIdx.x), slot = static_cast<int>(blockIdx.y);
  const int b = a.b0 + static_cast<int>(blockIdx.z);
  const int rem = slot * a.nchunks + c;
  const RowSlot rs = a.slot[slot];
  // the chunk's whole vectors: one TMA bulk copy; thread 0 waits (bounded,
  // sleeping between polls), the other threads at the barrier
  if (tid == 0) {
    if (a.trace)
      for (int k = 0; k < 7; ++k) sh.mk[k] = 0ull;
    mark(a, sh.mk, 0);
    const int e0 = c * a.chunk_elems;
    const int n = min(a.chunk_elems, a.V - e0);
    const uint32_t bulk = static_cast<uint32_t>((n * E::kSize) & ~15);
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&sh.bar, bulk);
    if (bulk)
      bulk_g2s(buf, row_ptr(a, rs.tensor, b, rs.row, E::kSize) + static_cast<int64_t>(e0) * E::kSize, bulk, &sh.bar);
    // tickets, taken while the copy is in flight: the last CTA of a pair to
    // start merges the pair, the last pair merger of a sequence to start
    // finishes the sequence.  Each waits only for CTAs that started before it.
    int role = 0;
    if (atomicAdd(pair_tkt(a, b, rs.row), 1u) + 1 == static_cast<uint32_t>(a.pair_chunks[rs.row])) {
      role = 1;
      if (a.do_verify && atomicAdd(seq_tkt(a, b), 1u) + 1 == static_cast<uint32_t>(a.npairs)) role = 2;
    }
    sh.flag = role;
    if (!mbar_wait_sleep(&sh.bar, 0)) {
      atomicOr(a.status, kFlagWaitTimeout);
      (void)mbar_wait_sleep(&sh.bar, 0);  // the copy still in flight: a second bounded wait before the buffer is read
    }
    mark(a, sh.mk, 1);
  }
  __syncthreads();
  const int role = sh.flag;
  stats_chunk<E>(a, b, slot, c, buf, sh);
  const int r = rs.row;
  __syncthreads();  // the chunk's records are written
  mark(a, sh.mk, 2);
  if (role == 0) {
    if (tid == 0) red_add_release(pair_pub(a, b, r), 1u);
  } else {
    // merge pair r once its other chunks are published
    if (tid == 0 && !wait_count(pair_pub(a, b, r), static_cast<uint32_t>(a.pair_chunks[r] - 1)))
      atomicOr(a.status, kFlagWaitTimeout);
    __syncthreads();
    mark(a, sh.mk, 3);
    Stage &st = *reinterpret_cast<Stage *>(buf);  // the chunk buffer is free again
    row_finish<E>(a, b, r, st, sh);
    mark(a, sh.mk, 4);
    if (a.do_verify) {
      __syncthreads();  // the pair's results are written
      if (role == 1) {
        if (tid == 0) red_add_release(seq_pub(a, b), 1u);
      } else {
        // a rejection the pair merges already resolved (ready word set) leaves
        // the sequence to the residual draw: nothing is left to finish here
        if (tid == 0) {
          sh.flag = (!a.greedy && ld_relaxed(ready_word(a, b)) != 0u) ? 1 : 0;
          if (!sh.flag && !wait_count(seq_pub(a, b), static_cast<uint32_t>(a.npairs - 1)))
            atomicOr(a.status, kFlagWaitTimeout);
        }
        __syncthreads();
        if (!sh.flag) seq_finish<E>(a, b, st, sh);
        mark(a, sh.mk, 5);
      }
    }
  }
  const int kind = role == 2 ? 3 : role;
  mark(a, sh.mk, 6);
  if (a.trace && tid == 0)
    trace_entry(a.trace + 8 * (static_cast<size_t>(b) * a.nslots * a.nchunks + rem), kind, b, rem, sh.mk);
}

// Thread 0 of a residual CTA: bounded wait (sleeping between polls) for a
// sequence's ready word; returns it (0: the wait ran out).  k_resid is a
// programmatic dependent launch that starts once every k_stats CTA has
// started, so the word is set unless k_stats failed.
SSD_DEV uint32_t wait_ready(const uint32_t *w) {
  for (uint32_t it = 0; it < kMaxPolls; ++it) {
    const uint32_t v = ld_relaxed(w);
    if (v) {
      fence_acq_rel();
      return v;
    }
    __nanosleep(500);
  }
  return 0u;
}

// Residual unit (sequence b, chunk c, quarter g = rounds 2g, 2g+1): once the
// sequence's acceptance chain has run, its block sums of max(0, p - q') over
// target and draft row a, read straight from global memory.  The unit with the
// sequence's last ticket draws the bonus once the others are published; it
// issues its staging loads before its own unit.  `rbst`: the sequence's
// residual block sums, staged for up to kResidStage chunks.
constexpr int kResidStage = 16;
template <class E>
SSD_DEV void resid_unit(const VocabArgs &a, float *umass, float *rbst, int32_t *pay, Smem &sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nu = a.nchunks * kQuarters;
  const int b = static_cast<int>(blockIdx.x / nu);
  const int u = static_cast<int>(blockIdx.x - static_cast<unsigned>(b) * nu);
  const int c = u / kQuarters, g = u % kQuarters;
  if (tid == 0) {
    const uint32_t v = wait_ready(ready_word(a, b));
    if (!v) atomicOr(a.status, kFlagWaitTimeout);
    const int acc0 = static_cast<int>(v) - 2;
    sh.flag = static_cast<int>(v);
    sh.ival[2] = (v && acc0 >= 0 && acc0 < a.K && atomicAdd(res_tkt(a, b), 1u) + 1 == static_cast<uint32_t>(nu)) ? 1 : 0;
  }
  __syncthreads();
  if (!sh.flag) return;
  const int acc = sh.flag - 2;
  if (acc < 0 || acc >= a.K) return;  // sequence finished in k_stats
  const bool fin = sh.ival[2] != 0;
  if (fin) stage_issue(a, b, pay, nullptr, false, sh);
  if (tid == 0 && a.trace)
    for (int k = 0; k < 7; ++k) sh.mk[k] = 0ull;
  mark(a, sh.mk, 0);
  const char *rowT = row_ptr(a, 0, b, acc, E::kSize);
  const char *rowD = row_ptr(a, 1, b, acc, E::kSize);
  {  // this lane's vectors of the unit, on their way into L1 while the row's statistics load
    const int e0 = c * a.chunk_elems;
    const int n = min(a.chunk_elems, a.V - e0);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int i0 = ((2 * g + jj) * kThreads + warp * 32 + lane) * E::kVec;
      if (i0 + E::kVec <= n) {
        const int64_t off = static_cast<int64_t>(e0 + i0) * E::kSize;
        asm volatile("prefetch.global.L1 [%0];" ::"l"(rowT + off));
        asm volatile("prefetch.global.L1 [%0];" ::"l"(rowD + off));
      }
    }
  }
  const size_t rr = static_cast<size_t>(b) * (a.K + 1) + acc;
  const RowInfo row = ldcg_row(a.rows + rr);
  const int F = a.Fs[acc];
  const uint64_t keyF = F > 0 ? ldcg_key(a.S + rr * a.Fcap + F - 1) : 0ull;
  const WResidual wf = residual_weights(a, row, keyF, F);
  float *rbs = a.rbs + (static_cast<size_t>(b) * a.nchunks + c) * kBlocks;
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int j = 2 * g + jj;
    float x[E::kVec];
    const float p = lane_weights<E, true, true>(a, rowT, rowD, c, j, warp, wf, x);
    const float incl = warp_incl_scan(p);
    if (lane == 31) {
      rbs[j * kWarps + warp] = incl;
      sh.bw[jj * kWarps + warp] = incl;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const float m = warp_total(sh.bw, 2 * kWarps);
    if (lane == 0) a.rmass[static_cast<size_t>(b) * nu + u] = m;
  }
  mark(a, sh.mk, 2);
  int kind = 2;
  __syncthreads();  // the unit's sums are written
  if (!fin) {
    if (tid == 0) red_add_release(res_pub(a, b), 1u);
  } else {
    kind = 3;
    if (tid == 0 && !wait_count(res_pub(a, b), static_cast<uint32_t>(nu - 1))) atomicOr(a.status, kFlagWaitTimeout);
    __syncthreads();
    mark(a, sh.mk, 3);
    // the unit masses and (up to kResidStage chunks) every unit's block sums
    for (int q = tid; q < nu; q += kThreads) cp_async4(&umass[q], a.rmass + static_cast<size_t>(b) * nu + q);
    const bool rbs_staged = a.nchunks <= kResidStage;
    if (rbs_staged) {
      const int4 *src = reinterpret_cast<const int4 *>(a.rbs + static_cast<size_t>(b) * a.nchunks * kBlocks);
      for (int i = tid; i < a.nchunks * (kBlocks / 4); i += kThreads) cp_async16(reinterpret_cast<int4 *>(rbst) + i, src + i);
    }
    const int acc2 = stage_complete(a, sh);  // the same chain: acc2 == acc
    const RowInfo ra = sh.rows[acc2];
    const WResidual wa = residual_weights(a, ra, sh.keyF[acc2], a.Fs[acc2]);
    const float ub = a.u_bonus[b];
    if (tid == 0) sh.near = 0;
    if (warp == 0) {
      locate(umass, nu, ub, false, sh);
      __syncwarp();
      const int uq = sh.ival[0];
      const float local = sh.scal[1];
      const float W = sh.scal[2];  // the residual's total mass
      __syncwarp();
      if (lane == 0) {
        sh.ival[6] = uq;
        sh.scal[6] = W;
      }
      if (uq >= 0) {
        const size_t o = (static_cast<size_t>(uq / kQuarters)) * kBlocks + 2 * (uq % kQuarters) * kWarps;
        if (lane < 2 * kWarps)
          sh.bw[lane] = rbs_staged ? rbst[o + lane] : __ldcg(a.rbs + static_cast<size_t>(b) * a.nchunks * kBlocks + o + lane);
        __syncwarp();
        locate(sh.bw, 2 * kWarps, local, true, sh);
        __syncwarp();
        if (lane == 0 && sh.ival[0] < 0) {  // a unit of positive mass has a positive block; kept for safety
          sh.ival[0] = 2 * kWarps - 1;
          sh.scal[1] = local;
          sh.near = 1;
        }
      }
    }
    __syncthreads();
    mark(a, sh.mk, 4);
    const int uq = sh.ival[6];
    const float W = sh.scal[6];
    int bt = -1;
    bool near = false;  // thread 0
    if (uq >= 0) {
      const int k = sh.ival[0];
      const float local2 = sh.scal[1];
      int d = -1;
      float dist = 0.f;
      if (warp == 0)
        d = warp_find<E, true, true>(a, rowT, rowD, uq / kQuarters, 2 * (uq % kQuarters) + k / kWarps, k % kWarps,
                                     local2, wa, &dist);
      __syncthreads();
      if (tid == 0) {
        sh.ival[4] = d;
        near = sh.near || !(dist >= __fmul_rn(kNearTie, W));
      }
      __syncthreads();
      bt = sh.ival[4];
    }
    const bool zero = uq < 0;  // no residual mass: p_{a+1} instead
    if (bt < 0) {
      bt = draw_target<E>(a, b, acc2, ra, ub, nullptr, sh);
      near = tid == 0 && sh.near;
    }
    if (a.do_lookup) {
      // the lookup lists, once the pair merge of position acc has written its list
      if (tid == 0 && !wait_count(pos_verdict(a, b, acc), 3u)) atomicOr(a.status, kFlagWaitTimeout);
      __syncthreads();
      stage_lists(a, b, sh);
      cp_async_wait_all();
      __syncthreads();
    }
    mark(a, sh.mk, 5);
    emit(a, b, acc2, bt, W, zero, near, pay, sh);
  }
  mark(a, sh.mk, 6);
  if (a.trace && tid == 0) {
    const size_t base = static_cast<size_t>(a.B) * a.nslots * a.nchunks;
    trace_entry(a.trace + 8 * (base + blockIdx.x), kind, b, u, sh.mk);
  }
}

template <class E>
__global__ void __launch_bounds__(kThreads, 4) k_resid(const __grid_constant__ VocabArgs a) {
  __shared__ Smem sh;
  __shared__ float umass[kMaxChunks * kQuarters];  // the sequence's unit masses (final draw)
  __shared__ int32_t pay[kPayStage];                // the sequence's cache payload (final draw)
  __shared__ __align__(16) float rbst[kResidStage * kBlocks];  // the sequence's residual block sums (final draw)
  resid_unit<E>(a, umass, rbst, pay, sh);
  // the grid completes only after k_stats has: its first CTA waits for it
  // before exiting
  if (blockIdx.x == 0 && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ===========================================================================
// round analytics: alpha_j, W_j, P(a = k), the hit rate, expected tokens
// ===========================================================================
// One CTA per (sequence b, position j = r + 1, unit u = chunk u / kQuarters,
// rounds 2 (u % kQuarters) and the next) of row pair r < K, once the
// statistics pass has merged the rows: the unit's sums of min(p, q') and of
// max(0, p - q') (each lane in element order, then the warps by a fixed tree).
template <class E>
__global__ void __launch_bounds__(kThreads) k_alpha(const __grid_constant__ VocabArgs a) {
  __shared__ float red[2][kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nu = a.nchunks * kQuarters;
  const long id = blockIdx.x;
  const int u = static_cast<int>(id % nu);
  const int r = static_cast<int>((id / nu) % a.K);
  const int b = static_cast<int>(id / (static_cast<long>(nu) * a.K));
  const size_t rr = static_cast<size_t>(b) * (a.K + 1) + r;
  const RowInfo ri = ldcg_row(a.rows + rr);
  const int F = a.Fs[r];
  const uint64_t keyF = F > 0 ? ldcg_key(a.S + rr * a.Fcap + F - 1) : 0ull;
  const WResidual wf = residual_weights(a, ri, keyF, F);  // p and q' factors
  const char *rowT = row_ptr(a, 0, b, r, E::kSize);
  const char *rowD = row_ptr(a, 1, b, r, E::kSize);
  const int c = u / kQuarters, g = u % kQuarters;
  const int e0 = c * a.chunk_elems;
  const int n = min(a.chunk_elems, a.V - e0);
  float smin = 0.f, sres = 0.f;
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int i0 = ((2 * g + jj) * kThreads + warp * 32 + lane) * E::kVec;
    float ft[E::kVec], fd[E::kVec];
    ld_vec<E>(rowT, e0, n, i0, -__int_as_float(0x7f800000), ft);
    ld_vec<E>(rowD, e0, n, i0, -__int_as_float(0x7f800000), fd);
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) {
      if (i0 + e >= n) continue;
      const float p = __fmul_rn(ex2(__fmaf_rn(ft[e], wf.kT, -wf.mtk)), wf.inv_st);
      const float f = (wf.hasS && cand_key(fd[e], e0 + i0 + e) >= wf.keyF) ? wf.fC : wf.f1;
      const float q = __fmul_rn(ex2(__fmaf_rn(fd[e], wf.kT, -wf.mdk)), f);
      smin = __fadd_rn(smin, fminf(p, q));
      sres = __fadd_rn(sres, fmaxf(__fsub_rn(p, q), 0.f));
    }
  }
  smin = warp_sum(smin);
  sres = warp_sum(sres);
  if (lane == 0) {
    red[0][warp] = smin;
    red[1][warp] = sres;
  }
  __syncthreads();
  if (tid == 0) {
    float m = 0.f, w = 0.f;
    for (int k = 0; k < kWarps; ++k) {
      m = __fadd_rn(m, red[0][k]);
      w = __fadd_rn(w, red[1][k]);
    }
    float *o = a.amass + ((static_cast<size_t>(b) * a.K + r) * nu + u) * 2;
    o[0] = m;
    o[1] = w;
  }
}

// One CTA per sequence, after k_alpha (T > 0) or straight after the
// statistics pass (T = 0, where p and q' are one-hot at the argmaxes): alpha
// and W per position, the chance that the bonus lands among the depth-k
// guesses given a = k, P(a = k), the hit rate and the expected tokens.
template <class E>
__global__ void __launch_bounds__(kThreads) k_analytics(const __grid_constant__ VocabArgs a) {
  __shared__ float s_alpha[kMaxK + 1], s_w[kMaxK + 1], s_hit[kMaxK + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int nu = a.nchunks * kQuarters;
  const int K = a.K;
  // alpha_j and W_j: warp r % kWarps sums position r's units in order
  for (int r = warp; r < K; r += kWarps) {
    const size_t rr = static_cast<size_t>(b) * (K + 1) + r;
    float al, w;
    if (a.greedy) {
      const RowInfo ri = ldcg_row(a.rows + rr);
      al = (ri.at == ri.ad) ? 1.f : 0.f;
      w = 1.f - al;
    } else {
      const float *m = a.amass + (static_cast<size_t>(b) * K + r) * nu * 2;
      float sa = 0.f, sw = 0.f;
      for (int u = lane; u < nu; u += 32) {
        sa = __fadd_rn(sa, __ldcg(m + 2 * u));
        sw = __fadd_rn(sw, __ldcg(m + 2 * u + 1));
      }
      al = warp_sum(sa);
      w = warp_sum(sw);
    }
    if (lane == 0) {
      s_alpha[r] = al;
      s_w[r] = w;
    }
  }
  __syncthreads();
  // hit masses: warp k % kWarps over depth k's guesses (S_{k+1}, the top-F_k
  // of draft row k), each weighted by the bonus distribution given a = k
  for (int k = warp; k <= K; k += kWarps) {
    const size_t rr = static_cast<size_t>(b) * (K + 1) + k;
    const RowInfo ri = ldcg_row(a.rows + rr);
    const int F = a.Fs[k];
    const char *rowT = row_ptr(a, 0, b, k, E::kSize);
    const bool resid = k < K && s_w[k] > 0.f;
    float h = 0.f;
    if (a.greedy) {
      // the bonus is the target argmax (the residual of one-hot rows is that
      // same one-hot whenever it has mass)
      for (int i = lane; i < F; i += 32)
        if (cand_idx(ldcg_key(a.S + rr * a.Fcap + i)) == ri.at) h = 1.f;
      h = warp_max(h);
    } else {
      const float mtk = __fmul_rn(ri.mt, a.kT);
      const float inv_st = __frcp_rn(ri.st);
      const float mdk = __fmul_rn(ri.md, a.kT);
      const float sN = __fmul_rn(ri.sd, norm_N(a.C, ri.sq));
      const float fC = __fdiv_rn(a.C, sN);
      for (int i = lane; i < F; i += 32) {
        const uint64_t key = ldcg_key(a.S + rr * a.Fcap + i);
        if (!key) continue;
        const int d = cand_idx(key);
        const float p = __fmul_rn(ex2(__fmaf_rn(E::ld(rowT, d), a.kT, -mtk)), inv_st);
        float x = p;
        if (resid) {  // every guess is in S, so q' carries the factor C
          const float q = __fmul_rn(ex2(__fmaf_rn(cand_val(key), a.kT, -mdk)), fC);
          x = fmaxf(__fsub_rn(p, q), 0.f);
        }
        h = __fadd_rn(h, x);
      }
      h = warp_sum(h);
      if (resid) h = __fdiv_rn(h, s_w[k]);
    }
    if (lane == 0) s_hit[k] = h;
  }
  __syncthreads();
  if (tid == 0) {
    float run = 1.f, hit = 0.f, etok = 0.f;
    for (int k = 0; k <= K; ++k) {
      const float pk = (k < K) ? __fmul_rn(run, s_w[k]) : run;
      if (k < K) run = __fmul_rn(run, s_alpha[k]);
      hit = __fmaf_rn(pk, s_hit[k], hit);
      etok = __fmaf_rn(pk, static_cast<float>(k + 1), etok);
      a.an_p_accept[static_cast<size_t>(b) * (K + 1) + k] = pk;
      if (a.an_hit_mass) a.an_hit_mass[static_cast<size_t>(b) * (K + 1) + k] = s_hit[k];
      if (k < K) {
        if (a.an_alpha) a.an_alpha[static_cast<size_t>(b) * K + k] = s_alpha[k];
        if (a.an_resid_w) a.an_resid_w[static_cast<size_t>(b) * K + k] = s_w[k];
      }
    }
    a.an_hit_rate[b] = hit;
    a.an_exp_tokens[b] = etok;
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
  int nslots, nchunks, chunk_elems, Fcap;
  size_t ctr_words;
  size_t ctr_off, stats_off, blk_off, bmk_off, rows_off, S_off, pos_off, rmass_off, rbs_off, amass_off, total;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int esize(ssd_dtype_t dt) { return dt == SSD_F32 ? 4 : 2; }

bool make_layout(int B, int K, int V, ssd_dtype_t dt, const int32_t *F, Layout *L) {
  if (B < 0 || K < 0 || K > kMaxK || V < 1 || !F) return false;
  if (dt != SSD_F32 && dt != SSD_BF16) return false;
  int fmax = 0;
  for (int k = 0; k <= K; ++k) {
    if (F[k] < 0 || F[k] > kMaxF || F[k] > V) return false;
    fmax = F[k] > fmax ? F[k] : fmax;
  }
  L->nslots = 2 * (K + 1);
  L->chunk_elems = kChunkBytes / esize(dt);
  L->nchunks = (V + L->chunk_elems - 1) / L->chunk_elems;
  if (L->nchunks > kMaxChunks) return false;
  L->Fcap = fmax > 0 ? fmax : 1;
  const size_t Bn = static_cast<size_t>(B > 0 ? B : 1);
  const size_t nrec = Bn * L->nslots * L->nchunks;
  L->ctr_words = ctr_words(Bn, K);
  size_t o = 0;
  L->ctr_off = o;
  o = align_up(o + L->ctr_words * sizeof(uint32_t), 256);
  L->stats_off = o;
  o = align_up(o + nrec * sizeof(ChunkStat), 256);
  L->blk_off = o;
  o = align_up(o + nrec * sizeof(BlockRec), 256);
  L->bmk_off = o;
  o = align_up(o + nrec * kBlocks * sizeof(uint32_t), 256);
  L->rows_off = o;
  o = align_up(o + Bn * (K + 1) * sizeof(RowInfo), 256);
  L->S_off = o;
  o = align_up(o + Bn * (K + 1) * L->Fcap * sizeof(uint64_t), 256);
  L->pos_off = o;
  o = align_up(o + Bn * (K > 0 ? K : 1) * sizeof(PosInfo), 256);
  L->rmass_off = o;
  o = align_up(o + Bn * L->nchunks * kQuarters * sizeof(float), 256);
  L->rbs_off = o;
  o = align_up(o + Bn * L->nchunks * kBlocks * sizeof(float), 256);
  L->amass_off = o;
  o = align_up(o + Bn * (K > 0 ? K : 1) * L->nchunks * kQuarters * 2 * sizeof(float), 256);
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
  a.nchunks = L.nchunks;
  a.chunk_elems = L.chunk_elems;
  a.Fcap = L.Fcap;
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
  a.stats = reinterpret_cast<ChunkStat *>(w + L.stats_off);
  a.bmk = reinterpret_cast<uint32_t *>(w + L.bmk_off);
  a.rows = reinterpret_cast<RowInfo *>(w + L.rows_off);
  a.S = reinterpret_cast<uint64_t *>(w + L.S_off);
  a.pos = reinterpret_cast<PosInfo *>(w + L.pos_off);
  a.blk = reinterpret_cast<BlockRec *>(w + L.blk_off);
  a.rmass = reinterpret_cast<float *>(w + L.rmass_off);
  a.rbs = reinterpret_cast<float *>(w + L.rbs_off);
  a.amass = reinterpret_cast<float *>(w + L.amass_off);
  a.status = status;
  return a;
}

// Rows read by a call: target rows 0..ntarget-1 and draft rows 0..ndraft-1,
// slots ordered by pair (target r, then draft r).  `topf`: draft rows keep
// their top-F_r lists.
void set_slots(VocabArgs &a, int ntarget, int ndraft, bool topf, bool draws) {
  int n = 0;
  a.npairs = ntarget > ndraft ? ntarget : ndraft;
  for (int r = 0; r <= a.K; ++r) {
    a.tsl[r] = a.dsl[r] = -1;
    a.pair_chunks[r] = 0;
    a.Fs[r] = (topf && r < ndraft) ? a.F[r] : 0;
  }
  for (int r = 0; r < a.npairs; ++r) {
    int rows = 0;
    if (r < ntarget) {
      a.tsl[r] = n;
      // block sums on the rows a draw may use: target row K (the bonus after
      // full acceptance) and the draft rows sampled from (d_{r+1})
      const bool blk = draws && a.do_verify && r == a.K;
      a.slot[n++] = RowSlot{0, static_cast<int16_t>(r), 0, static_cast<int16_t>(blk)};
      ++rows;
    }
    if (r < ndraft) {
      a.dsl[r] = n;
      const bool blk = draws && a.do_sample && r < a.K;
      a.slot[n++] = RowSlot{1, static_cast<int16_t>(r), static_cast<int16_t>(a.Fs[r]), static_cast<int16_t>(blk)};
      ++rows;
    }
    a.pair_chunks[r] = rows * a.nchunks;
  }
  a.nslots = n;
}

// Optional timing hook (ssd_set_timing_events): events recorded around the
// statistics kernel of every vocabulary call while set.
cudaEvent_t g_ev_before = nullptr;
cudaEvent_t g_ev_after = nullptr;
// Optional per-CTA trace (ssd_set_trace).
void *g_trace = nullptr;
size_t g_trace_bytes = 0;

constexpr size_t kStatsSmem = kChunkBytes + sizeof(Smem);
static_assert(kStatsCtas * (kStatsSmem + 1024) <= 228 * 1024, "shared memory of k_stats too large for its CTAs/SM");

ssd_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_smem_attr_set[2][kMaxDevices / 64 + 1];

template <class E>
cudaError_t launch_vocab(VocabArgs &a, cudaStream_t s) {
  constexpr int ti = E::kSize == 4 ? 0 : 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const uint64_t bit = 1ull << (dev % 64);
  if (!(g_smem_attr_set[ti][dev / 64].load() & bit)) {
    e = cudaFuncSetAttribute(k_stats<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kStatsSmem));
    if (e != cudaSuccess) return e;
    g_smem_attr_set[ti][dev / 64].fetch_or(bit);
  }
  const long n1 = static_cast<long>(a.B) * a.nslots * a.nchunks;
  const long n2 = (a.do_verify && !a.greedy && a.K > 0) ? static_cast<long>(a.B) * a.nchunks * kQuarters : 0;
  if (n1 < 1) return cudaSuccess;
  if (n1 > 0x7fffffffL) return cudaErrorInvalidValue;
  a.nst = n1;
  a.trace = (g_trace && g_trace_bytes >= static_cast<size_t>(n1 + n2) * 64)
                ? static_cast<unsigned long long *>(g_trace)
                : nullptr;
  // counters start at zero
  e = cudaMemsetAsync(a.ctr, 0, ctr_words(static_cast<size_t>(a.B), a.K) * sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  if (g_ev_before) cudaEventRecord(g_ev_before, s);
  // grid (chunk, row slot, sequence); sequences in launches of at most 65535
  for (int b0 = 0; b0 < a.B; b0 += 65535) {
    a.b0 = b0;
    const unsigned nb = static_cast<unsigned>(a.B - b0 < 65535 ? a.B - b0 : 65535);
    k_stats<E><<<dim3(static_cast<unsigned>(a.nchunks), static_cast<unsigned>(a.nslots), nb), kThreads, kStatsSmem,
                 s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  a.b0 = 0;
  if (g_ev_after) cudaEventRecord(g_ev_after, s);
  if (n2 > 0) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(n2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_resid<E>, a);
  }
  return e;
}

cudaError_t launch_any(ssd_dtype_t dt, VocabArgs &a, cudaStream_t s) {
  return dt == SSD_F32 ? launch_vocab<EF32>(a, s) : launch_vocab<EBF16>(a, s);
}

// The analytics kernels after the statistics pass: the unit sums of every
// row pair r < K (T > 0), then one CTA per sequence.
template <class E>
cudaError_t launch_analytics(const VocabArgs &a, cudaStream_t s) {
  if (a.B < 1) return cudaSuccess;
  if (!a.greedy && a.K > 0) {
    const long n = static_cast<long>(a.B) * a.K * a.nchunks * kQuarters;
    if (n > 0x7fffffffL) return cudaErrorInvalidValue;
    k_alpha<E><<<static_cast<unsigned>(n), kThreads, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  k_analytics<E><<<static_cast<unsigned>(a.B), kThreads, 0, s>>>(a);
  return cudaGetLastError();
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
  set_slots(a, 0, K, C < 1.f, !a.greedy);
  a.u_draft = u_draft;
  a.d_out = d_out;
  a.qd_out = qd_out;
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
  set_slots(a, K + 1, K, C < 1.f, !a.greedy);
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
  set_slots(a, 0, K + 1, true, false);
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

ssd_status_t ssd_round(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                       int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                       const float *u_draft, const float *u_acc, const float *u_bonus, const int32_t *payload,
                       int32_t *d_out, float *qd_out, int32_t *accept_len, int32_t *out_tokens, int32_t *bonus,
                       float *accept_prob, float *resid_mass, int32_t *guess, float *guess_q, int32_t *slot,
                       int32_t *next_tokens, uint32_t *hits, uint32_t *near_ties, uint32_t *status, void *ws,
                       size_t ws_bytes, ssd_stream_t s) {
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
  set_slots(a, K + 1, a.do_predict ? K + 1 : K, a.do_predict || C < 1.f, !a.greedy);
  a.u_draft = u_draft;
  a.u_acc = u_acc;
  a.u_bonus = u_bonus;
  a.payload = payload;
  a.d_out = d_out;
  a.qd_out = qd_out;
  a.d_in = d_out;
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
  return cuda_status(launch_any(dt, a, cs));
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
  set_slots(a, K + 1, K + 1, true, false);
  a.an_alpha = alpha;
  a.an_resid_w = resid_w;
  a.an_p_accept = p_accept;
  a.an_hit_mass = hit_mass;
  a.an_hit_rate = hit_rate;
  a.an_exp_tokens = exp_tokens;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  cudaError_t e = launch_any(dt, a, cs);
  if (e == cudaSuccess) e = dt == SSD_F32 ? launch_analytics<EF32>(a, cs) : launch_analytics<EBF16>(a, cs);
  return cuda_status(e);
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
