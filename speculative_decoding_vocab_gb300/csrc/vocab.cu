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
// Structure: every vocabulary call is ONE persistent kernel, k_vocab, fed by a
// global work queue (an atomic counter).  Work items, in queue order:
//   STATS(b, slot, chunk)  the HBM pass: a 32 KiB chunk of one logit row is
//                          staged in shared memory by a TMA bulk copy and
//                          reduced to (max, sum of 2^(z log2e/T - max), argmax,
//                          sorted top-F candidates).  >= 95% of the bytes.
//   ROW(b, r)              merges row r's chunk records (target and draft),
//                          Saguaro-samples d_{r+1} (locate the chunk from the
//                          chunk masses, rescan only that chunk), gathers
//                          p(d), q'(d), writes the guesses of depth r.
//   RES(b, c)              acceptance chain, then the residual mass of chunk c
//                          of row a (the rejected position).
//   FIN(b)                 residual / bonus draw (locate the chunk, rescan it),
//                          outputs, cache lookup.
// Each group of sequence b is queued a few sequences after its inputs, and an
// item only ever waits (bounded, on a per-sequence counter) for items EARLIER
// in the queue.  Items are dequeued in index order by running CTAs, so every
// awaited item is held by a running CTA: the schedule cannot deadlock, with or
// without co-residency of the grid.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/ssd.h"
#include "common.cuh"

namespace ssd {

constexpr int kThreads = 256;
constexpr int kChunkBytes = 24576;  // = kThreads * kSegVec * 16 B
constexpr int kStages = 3;
constexpr int kCandCap = 512;
constexpr int kMaxK = 16;
constexpr int kMaxSlots = 2 * (kMaxK + 1);
constexpr int kMaxF = 256;
constexpr int kMaxChunks = 128;  // per row: 4 lists per lane in the warp merge
constexpr uint32_t kMaxSpins = 1u << 24;  // bounded dependency waits (x ~100 ns sleeps)

enum ItemKind { IT_STATS = 0, IT_ROW = 1, IT_RES = 2, IT_FIN = 3, IT_NONE = 4 };

struct ChunkStat {
  float m;   // chunk maximum
  float s;   // sum over the chunk of 2^(z kT - fl(m kT)) (0 when greedy)
  int amax;  // lowest index holding m
  int pad;
};
struct RowSlot {
  int16_t tensor;  // 0 = target, 1 = draft
  int16_t row;
  int16_t F;  // top-F candidates wanted (0 = none)
  int16_t pad;
};
struct RowInfo {  // merged statistics of row r of a sequence
  float mt, st;   // target max, sum relative to fl(mt kT)
  int at, pad0;   // target argmax
  float md, sd;   // draft max, sum
  int ad;         // draft argmax
  float sq;       // sum of q over S (normalised)
};
struct PosInfo {  // draft token d_j and its probabilities
  int d;
  float p, q;  // p_j(d), q'_j(d); p < 0 marks an invalid token
  int pad;
};
struct ResInfo {
  float w;   // residual mass of a chunk of row a
  int last;  // last index of the chunk with positive residual (-1: none)
};

struct Sched {
  int B, ns, nr, nc, nf;  // items per sequence: stats, row, residual, final
  int L1, L2, L3;         // lags of the row / residual / final groups (in sequences)
};

struct VocabArgs {
  const void *target, *draft;
  int64_t seq_stride, row_stride;  // elements
  int B, K, V;
  int nslots, nchunks, chunk_elems, Fcap;
  float kT;    // log2(e) / T
  int greedy;  // T == 0
  float C;
  int tslot0, dslot0;  // slot of target row 0 (-1: no target rows) and draft row 0
  int do_sample, do_verify, do_predict, do_lookup;
  RowSlot slot[kMaxSlots];
  int F[kMaxK + 1];
  int foff[kMaxK + 2];
  Sched fs;   // finish queue: super-slot t holds ROW(t), RES(t-1), FIN(t-2); fs.ns = statistics per sequence
  long nst;   // statistics items in total (B * fs.ns)
  // workspace
  uint32_t *ctr;  // [0] queue head, [1] abort, [2] finished sequences, [3] hits; 3 per sequence after
  ChunkStat *stats;
  uint64_t *cands;  // [B][nslots][nchunks][Fcap]
  RowInfo *rows;    // [B][K+1]
  uint64_t *S;      // [B][K+1][Fcap] merged top-F lists
  PosInfo *pos;     // [B][K]
  ResInfo *res;     // [B][nchunks]
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
  uint32_t *status;
  unsigned long long *trace;  // optional: 4 words per queue entry (see ssd_set_trace)
};

SSD_DEV uint32_t *stats_done(const VocabArgs &a, int b) { return a.ctr + 4 + 3 * b; }
SSD_DEV uint32_t *row_done(const VocabArgs &a, int b) { return a.ctr + 5 + 3 * b; }
SSD_DEV uint32_t *res_done(const VocabArgs &a, int b) { return a.ctr + 6 + 3 * b; }

__host__ __device__ inline size_t chunk_index(const VocabArgs &a, int b, int slot, int c) {
  return (static_cast<size_t>(b) * a.nslots + slot) * a.nchunks + c;
}
SSD_DEV const char *row_ptr(const VocabArgs &a, int tensor, int b, int row, int esize) {
  const char *base = reinterpret_cast<const char *>(tensor ? a.draft : a.target);
  return base + (static_cast<int64_t>(b) * a.seq_stride + static_cast<int64_t>(row) * a.row_stride) * esize;
}

// ---------------------------------------------------------------------------
// finish queue: super-slot t holds ROW(t - L1), RES(t - L2), FIN(t - L3)
// ---------------------------------------------------------------------------
__host__ __device__ inline long clampi(long x, long lo, long hi) { return x < lo ? lo : (x > hi ? hi : x); }
__host__ __device__ inline long sched_start(const Sched &s, long t) {
  return s.nr * clampi(t - s.L1, 0, s.B) + s.nc * clampi(t - s.L2, 0, s.B) + s.nf * clampi(t - s.L3, 0, s.B);
}
__host__ __device__ inline long sched_total(const Sched &s) { return sched_start(s, s.B + s.L3); }

SSD_DEV void sched_decode(const Sched &s, long q, int &kind, int &b, int &idx) {
  long lo = 0, hi = s.B + s.L3;  // the super-slot t with start(t) <= q < start(t+1)
  while (hi - lo > 1) {
    const long mid = (lo + hi) >> 1;
    if (sched_start(s, mid) <= q) lo = mid;
    else hi = mid;
  }
  const long t = lo;
  long off = q - sched_start(s, t);
  if (t - s.L1 >= 0 && t - s.L1 < s.B) {
    if (off < s.nr) {
      kind = IT_ROW;
      b = static_cast<int>(t - s.L1);
      idx = static_cast<int>(off);
      return;
    }
    off -= s.nr;
  }
  if (t - s.L2 >= 0 && t - s.L2 < s.B) {
    if (off < s.nc) {
      kind = IT_RES;
      b = static_cast<int>(t - s.L2);
      idx = static_cast<int>(off);
      return;
    }
    off -= s.nc;
  }
  kind = IT_FIN;
  b = static_cast<int>(t - s.L3);
  idx = 0;
}

// ---------------------------------------------------------------------------
// dependency counters
// ---------------------------------------------------------------------------
SSD_DEV uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// shared memory of the persistent CTA
// ---------------------------------------------------------------------------
struct Smem {
  float wm[kThreads / 32], ws[kThreads / 32];
  int wa[kThreads / 32];
  float red[kThreads / 32 + 1];
  uint64_t redk[kThreads / 32];
  int ncand;
  int item_kind[2], item_b[2], item_idx[2], item_stage[2];
  long item_q[2];
  int ok;
  int found, last_pos;
  float scal[8];
  int ival[8];
  RowInfo ri;
  float cmass[kMaxChunks];
  ChunkStat cs[2][kMaxChunks];
  uint64_t S[kMaxF];
  float cp[kMaxK], cq[kMaxK], cu[kMaxK];
};

// All threads call after writing an item's results; thread 0 publishes.
SSD_DEV void signal_done(uint32_t *ctr) {
  group_sync<kThreads>();  // every thread's writes of the item precede thread 0's release
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}

// ===========================================================================
// STATS item
// ===========================================================================
template <class E>
SSD_DEV void issue_stats(const VocabArgs &a, int b, int idx, uint8_t *dst, uint64_t *bar) {
  const int slot = idx / a.nchunks, c = idx % a.nchunks;
  const RowSlot rs = a.slot[slot];
  const int e0 = c * a.chunk_elems;
  const int n = min(a.chunk_elems, a.V - e0);
  const uint32_t bulk = static_cast<uint32_t>((n * E::kSize) & ~15);
  const char *src = row_ptr(a, rs.tensor, b, rs.row, E::kSize) + static_cast<int64_t>(e0) * E::kSize;
  mbar_arrive_expect_tx(bar, bulk);
  if (bulk) bulk_g2s(dst, src, bulk, bar);
}

// A thread's running state over its groups (16-byte vectors, or the one tail
// element): maximum m1 and the group holding it, the second-largest group
// maximum m2, and the sum of 2^(z kT - mk) with mk = fl(m1 kT).
struct Stream {
  float m1, m2, s, mk;
  int g1;
};

template <int N>
SSD_DEV void stream_update(Stream &st, const float *f, int g, float kT, bool greedy) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  float vm = f[0];
#pragma unroll
  for (int e = 1; e < N; ++e) vm = fmaxf(vm, f[e]);
  if (vm > st.m2) {
    if (vm > st.m1) {
      st.m2 = st.m1;
      if (!greedy) {
        const float nk = __fmul_rn(vm, kT);
        if (st.m1 != NEG_INF) st.s = __fmul_rn(st.s, ex2(__fsub_rn(st.mk, nk)));
        st.mk = nk;
      }
      st.m1 = vm;
      st.g1 = g;
    } else {
      st.m2 = vm;
    }
  }
  if (!greedy && st.m1 != NEG_INF) {
#pragma unroll
    for (int e = 0; e < N; ++e) st.s = __fadd_rn(st.s, ex2(__fmaf_rn(f[e], kT, -st.mk)));
  }
}

template <class E>
SSD_DEV void stats_item(const VocabArgs &a, int b, int idx, const uint8_t *buf, uint64_t *cand, Smem &sh) {
  constexpr int NT = kThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = idx / a.nchunks, c = idx % a.nchunks;
  const RowSlot rs = a.slot[slot];
  const int e0 = c * a.chunk_elems;
  const int n = min(a.chunk_elems, a.V - e0);
  const int nvec = (n * E::kSize) >> 4;
  const int nbulk = nvec * E::kVec;
  const int ntail = n - nbulk;  // < kVec elements, only in a row's last chunk
  const char *row = row_ptr(a, rs.tensor, b, rs.row, E::kSize);
  const uint4 *v4 = reinterpret_cast<const uint4 *>(buf);
  const float kT = a.kT;
  const bool greedy = a.greedy != 0;
  const float NEG_INF = -__int_as_float(0x7f800000);

  // ---- stream: thread t owns vectors t, t+NT, ...; tail element i belongs to thread i
  Stream st{NEG_INF, NEG_INF, 0.f, 0.f, -1};
  for (int v = tid; v < nvec; v += NT) {
    float f[E::kVec];
    E::unpack(v4[v], f);
    stream_update<E::kVec>(st, f, v, kT, greedy);
  }
  const float zt = (tid < ntail) ? E::ld(row, e0 + nbulk + tid) : NEG_INF;
  if (tid < ntail) stream_update<1>(st, &zt, nvec, kT, greedy);
  // chunk-local index of the thread's first maximum (within group g1)
  int tidx = 0x7fffffff;
  if (st.g1 >= 0) {
    if (st.g1 < nvec) {
      float f[E::kVec];
      E::unpack(v4[st.g1], f);
#pragma unroll
      for (int e = E::kVec - 1; e >= 0; --e)
        if (f[e] == st.m1) tidx = st.g1 * E::kVec + e;
    } else {
      tidx = nbulk + tid;
    }
  }
  // ---- per warp: max, sum rescaled to it, lowest argmax
  float wm = st.m1;
#pragma unroll
  for (int o = 16; o; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
  float sr = 0.f;
  if (!greedy && st.m1 != NEG_INF) sr = __fmul_rn(st.s, ex2(__fsub_rn(st.mk, __fmul_rn(wm, kT))));
  sr = warp_sum(sr);
  int wi = (st.m1 == wm) ? tidx : 0x7fffffff;
#pragma unroll
  for (int o = 16; o; o >>= 1) wi = min(wi, __shfl_xor_sync(0xffffffffu, wi, o));
  if (lane == 0) {
    sh.wm[warp] = wm;
    sh.ws[warp] = sr;
    sh.wa[warp] = wi;
  }
  const int F = rs.F;
  const uint32_t mykey = (st.g1 >= 0) ? f2ord(st.m1) : 0u;
  uint32_t tau = 0;
  if (F > 1) {
    // tau: the F-th largest per-thread maximum; at least F elements reach it
    for (int bit = 31; bit >= E::kLowBit; --bit) {
      const uint32_t t = tau | (1u << bit);
      if (group_sync_count<kThreads>(mykey >= t) >= F) tau = t;
    }
    if (tid == 0) sh.ncand = 0;
  }
  group_sync<kThreads>();
  float M = sh.wm[0];
  for (int w = 1; w < NT / 32; ++w) M = fmaxf(M, sh.wm[w]);
  int amax = 0x7fffffff;
  for (int w = 0; w < NT / 32; ++w)
    if (sh.wm[w] == M) amax = min(amax, sh.wa[w]);
  uint64_t *out = a.cands + chunk_index(a, b, slot, c) * a.Fcap;
  if (F > 1) {
    // candidates: a thread whose second group maximum is below tau holds every
    // element >= tau in group g1; otherwise it rescans all of its groups
    if (mykey >= tau && st.g1 >= 0) {
      const bool one = (st.m2 == NEG_INF) || f2ord(st.m2) < tau;
      if (one) {
        if (st.g1 < nvec) {
          float f[E::kVec];
          E::unpack(v4[st.g1], f);
#pragma unroll
          for (int e = 0; e < E::kVec; ++e)
            if (f2ord(f[e]) >= tau) {
              const int p = atomicAdd(&sh.ncand, 1);
              if (p < kCandCap) cand[p] = cand_key(f[e], e0 + st.g1 * E::kVec + e);
            }
        } else {
          const int p = atomicAdd(&sh.ncand, 1);
          if (p < kCandCap) cand[p] = cand_key(zt, e0 + nbulk + tid);
        }
      } else {
        for (int g = tid; g < nvec; g += NT) {
          float f[E::kVec];
          E::unpack(v4[g], f);
#pragma unroll
          for (int e = 0; e < E::kVec; ++e)
            if (f2ord(f[e]) >= tau) {
              const int p = atomicAdd(&sh.ncand, 1);
              if (p < kCandCap) cand[p] = cand_key(f[e], e0 + g * E::kVec + e);
            }
        }
        if (tid < ntail && f2ord(zt) >= tau) {
          const int p = atomicAdd(&sh.ncand, 1);
          if (p < kCandCap) cand[p] = cand_key(zt, e0 + nbulk + tid);
        }
      }
    }
    group_sync<kThreads>();
    const int nc = sh.ncand;
    if (nc <= kCandCap) {
      int P = 1;
      while (P < nc || P < F) P <<= 1;
      for (int i = nc + tid; i < P; i += NT) cand[i] = 0ull;
      group_sync<kThreads>();
      if (P <= 64) {
        // one warp sorts in registers, descending: key i lives in lane i & 31, half i >> 5
        if (warp == 0) {
          uint64_t x[2];
          x[0] = (lane < P) ? cand[lane] : 0ull;
          x[1] = (lane + 32 < P) ? cand[lane + 32] : 0ull;
          for (int k = 2; k <= 64; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
              if (j == 32) {
                // partner of i is i + 32 in the same lane; k == 64: descending
                if (x[0] < x[1]) {
                  const uint64_t t = x[0];
                  x[0] = x[1];
                  x[1] = t;
                }
              } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int i = lane + 32 * h;
                  const uint64_t y = __shfl_xor_sync(0xffffffffu, x[h], j);
                  const bool desc = ((i & k) == 0);
                  const bool lower = ((i & j) == 0);
                  const bool keep_max = (desc == lower);
                  x[h] = keep_max ? (x[h] > y ? x[h] : y) : (x[h] < y ? x[h] : y);
                }
              }
            }
          }
          if (lane < F) out[lane] = x[0];
          if (lane + 32 < F) out[lane + 32] = x[1];
        }
      } else {
        for (int k = 2; k <= P; k <<= 1) {
          for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P; i += NT) {
              const int ixj = i ^ j;
              if (ixj > i) {
                const uint64_t x = cand[i], y = cand[ixj];
                const bool desc = (i & k) == 0;
                if (desc ? (x < y) : (x > y)) {
                  cand[i] = y;
                  cand[ixj] = x;
                }
              }
            }
            group_sync<kThreads>();
          }
        }
        for (int i = tid; i < F; i += NT) out[i] = cand[i];
      }
    } else {
      // too many ties at the threshold: exact selection, one winner per sweep
      uint64_t prev = ~0ull;
      for (int r = 0; r < F; ++r) {
        uint64_t best = 0;
        for (int g = tid; g < nvec; g += NT) {
          float f[E::kVec];
          E::unpack(v4[g], f);
#pragma unroll
          for (int e = 0; e < E::kVec; ++e) {
            const uint64_t key = cand_key(f[e], e0 + g * E::kVec + e);
            if (key < prev && key > best) best = key;
          }
        }
        if (tid < ntail) {
          const uint64_t key = cand_key(zt, e0 + nbulk + tid);
          if (key < prev && key > best) best = key;
        }
        best = block_max_u64<NT>(best, sh.redk);
        if (tid == 0) out[r] = best;
        prev = best;
      }
    }
  } else if (F == 1 && tid == 0) {
    out[0] = cand_key(M, e0 + (amax == 0x7fffffff ? 0 : amax));
  }
  if (tid == 0) {
    float S = 0.f;
    if (!greedy && M != NEG_INF) {
      const float Mk = __fmul_rn(M, kT);
      for (int w = 0; w < NT / 32; ++w)
        if (sh.wm[w] != NEG_INF)
          S = __fadd_rn(S, __fmul_rn(sh.ws[w], ex2(__fsub_rn(__fmul_rn(sh.wm[w], kT), Mk))));
    }
    ChunkStat cs;
    cs.m = M;
    cs.s = S;
    cs.amax = e0 + (amax == 0x7fffffff ? 0 : amax);  // an all -inf chunk: its first index
    cs.pad = 0;
    a.stats[chunk_index(a, b, slot, c)] = cs;
  }
  signal_done(stats_done(a, b));
}

// ===========================================================================
// merges (records are first copied to shared memory by all threads at once,
// so no thread walks a chain of dependent global loads)
// ===========================================================================
struct RowStat {
  float m, s;
  int amax;
};
// Chunks in index order: a strictly larger maximum keeps the lowest index.
SSD_DEV RowStat merge_row_smem(const VocabArgs &a, const ChunkStat *cs) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  RowStat r{cs[0].m, 0.f, cs[0].amax};
  for (int c = 1; c < a.nchunks; ++c)
    if (cs[c].m > r.m) {
      r.m = cs[c].m;
      r.amax = cs[c].amax;
    }
  if (!a.greedy && r.m != NEG_INF) {
    const float mk = __fmul_rn(r.m, a.kT);
    for (int c = 0; c < a.nchunks; ++c)
      if (cs[c].m != NEG_INF) r.s = __fadd_rn(r.s, __fmul_rn(cs[c].s, ex2(__fsub_rn(__fmul_rn(cs[c].m, a.kT), mk))));
  }
  return r;
}

// Warp-cooperative k-way merge of the sorted per-chunk candidate lists
// (list c at lists[c * stride], F keys each) into the top-F list `dst`
// (descending keys; sentinel 0 past the end).
SSD_DEV void merge_topf(const uint64_t *lists, size_t stride, int nchunks, int F, uint64_t *dst) {
  constexpr int L = kMaxChunks / 32;
  const int lane = threadIdx.x & 31;
  int ptr[L];
  uint64_t head[L];
#pragma unroll
  for (int l = 0; l < L; ++l) {
    const int c = lane + 32 * l;
    ptr[l] = 0;
    head[l] = (c < nchunks && F > 0) ? lists[c * stride] : 0ull;
  }
  for (int r = 0; r < F; ++r) {
    uint64_t best = 0;
    int bl = -1;
#pragma unroll
    for (int l = 0; l < L; ++l)
      if (head[l] > best) {
        best = head[l];
        bl = l;
      }
    const uint64_t win = warp_max_u64(best);
    if (lane == 0) dst[r] = win;
    if (win != 0 && best == win && bl >= 0) {
#pragma unroll
      for (int l = 0; l < L; ++l)
        if (l == bl) {
          const int c = lane + 32 * l;
          ++ptr[l];
          head[l] = (ptr[l] < F) ? lists[c * stride + ptr[l]] : 0ull;
        }
    }
  }
  __syncwarp();
}

// ===========================================================================
// inverse-CDF draws over one chunk of a row (one CTA)
// ===========================================================================
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

// A chunk is split into kThreads contiguous segments of kSegVec vectors; thread
// t owns elements [start + t*SEG, start + (t+1)*SEG).  Its segment sum is taken
// in index order, the segments are combined by one block-wide exclusive scan:
// that fixed order defines the chunk's running weights for both range_total
// and range_find.
constexpr int kSegVec = 6;
static_assert(kChunkBytes == kThreads * kSegVec * 16, "a chunk is one segment per thread");

// 16 raw bytes of a row at element i0; lanes at or past `end` are left zero
// (callers mask them by index).
template <class E>
SSD_DEV uint4 ld_raw(const char *row, int i0, int end) {
  if (i0 + E::kVec <= end) return __ldg(reinterpret_cast<const uint4 *>(row + static_cast<int64_t>(i0) * E::kSize));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  for (int e = 0; e < E::kVec && i0 + e < end; ++e) {
    if (E::kSize == 4) {
      w[e] = __ldg(reinterpret_cast<const uint32_t *>(row) + i0 + e);
    } else {
      const uint32_t h = __ldg(reinterpret_cast<const unsigned short *>(row) + i0 + e);
      w[e >> 1] |= h << ((e & 1) * 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// This thread's segment of one or two rows, loaded in one round of 16-byte loads.
template <class E>
struct Segment {
  uint4 t[kSegVec], d[kSegVec];
  SSD_DEV void load(const char *rowT, const char *rowD, int s0, int end) {
#pragma unroll
    for (int v = 0; v < kSegVec; ++v) {
      t[v] = rowT ? ld_raw<E>(rowT, s0 + v * E::kVec, end) : make_uint4(0, 0, 0, 0);
      d[v] = rowD ? ld_raw<E>(rowD, s0 + v * E::kVec, end) : make_uint4(0, 0, 0, 0);
    }
  }
  // sum of weights in index order; *last = last index with w > 0
  template <class WF>
  SSD_DEV float sum(int s0, int end, const WF &wf, int *last) const {
    float acc = 0.f;
#pragma unroll
    for (int v = 0; v < kSegVec; ++v) {
      float ft[E::kVec], fd[E::kVec];
      E::unpack(t[v], ft);
      E::unpack(d[v], fd);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) {
        const int i = s0 + v * E::kVec + e;
        const float x = (i < end) ? wf(ft[e], fd[e], i) : 0.f;
        acc = __fadd_rn(acc, x);
        if (x > 0.f) *last = i;
      }
    }
    return acc;
  }
  // first index whose running weight (offset by `base`) exceeds `target`, with w > 0; -1 if none
  template <class WF>
  SSD_DEV int find(int s0, int end, const WF &wf, float base, float target) const {
    float run = 0.f;
    int hit = -1;
#pragma unroll
    for (int v = 0; v < kSegVec; ++v) {
      float ft[E::kVec], fd[E::kVec];
      E::unpack(t[v], ft);
      E::unpack(d[v], fd);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) {
        const int i = s0 + v * E::kVec + e;
        const float x = (i < end) ? wf(ft[e], fd[e], i) : 0.f;
        run = __fadd_rn(run, x);
        if (hit < 0 && x > 0.f && __fadd_rn(base, run) > target) hit = i;
      }
    }
    return hit;
  }
};

// Total weight of [start, end) (end - start <= one chunk) in the segment order;
// *last = last index with w > 0 (-1 if none).
template <class E, class WF>
SSD_DEV float range_total(const char *rowT, const char *rowD, int start, int end, const WF &wf, int *last,
                          Smem &sh) {
  constexpr int SEG = kSegVec * E::kVec;
  const int tid = threadIdx.x;
  const int s0 = start + tid * SEG;
  Segment<E> seg;
  seg.load(rowT, rowD, s0, end);
  int lp = -1;
  const float t = seg.sum(s0, end, wf, &lp);
  if (tid == 0) sh.last_pos = -1;
  const float ex = block_excl_scan<kThreads>(t, sh.red);  // (contains barriers)
  if (tid == kThreads - 1) sh.scal[0] = __fadd_rn(ex, t);
  atomicMax(&sh.last_pos, lp);
  group_sync<kThreads>();
  const float tot = sh.scal[0];
  *last = sh.last_pos;
  group_sync<kThreads>();
  return tot;
}

// First i in [start, end) whose running weight from `start` (segment order as in
// range_total) exceeds `target` and whose weight is positive; -1 when none.
template <class E, class WF>
SSD_DEV int range_find(const char *rowT, const char *rowD, int start, int end, float target, const WF &wf,
                       Smem &sh) {
  constexpr int SEG = kSegVec * E::kVec;
  const int tid = threadIdx.x;
  const int s0 = start + tid * SEG;
  Segment<E> seg;
  seg.load(rowT, rowD, s0, end);
  int lp = -1;
  const float t = seg.sum(s0, end, wf, &lp);
  const float ex = block_excl_scan<kThreads>(t, sh.red);
  if (tid == 0) sh.found = 0x7fffffff;
  group_sync<kThreads>();
  // the segment where the running weight first exceeds the target (the earliest wins)
  if (t > 0.f && __fadd_rn(ex, t) > target) {
    int hit = seg.find(s0, end, wf, ex, target);
    if (hit < 0) hit = lp;  // rounding inside the segment: its last positive element
    atomicMin(&sh.found, hit);
  }
  group_sync<kThreads>();
  const int r = sh.found;
  group_sync<kThreads>();
  return r == 0x7fffffff ? -1 : r;
}

// Locate the chunk holding u * W among per-chunk masses sh.cmass[0..nchunks)
// (summed in chunk order) -- thread 0 -- with the target inside that chunk.
SSD_DEV void locate_chunk(int nchunks, float u, Smem &sh) {
  if (threadIdx.x == 0) {
    float W = 0.f;
    for (int c = 0; c < nchunks; ++c) W = __fadd_rn(W, sh.cmass[c]);
    const float target = __fmul_rn(u, W);
    int cs = -1;
    float before = 0.f, cum = 0.f;
    for (int c = 0; c < nchunks; ++c) {
      const float nc = __fadd_rn(cum, sh.cmass[c]);
      if (nc > target && sh.cmass[c] > 0.f) {
        cs = c;
        before = cum;
        break;
      }
      cum = nc;
    }
    if (cs < 0 && W > 0.f)  // rounding left u * W past the end: the last chunk with mass
      for (int c = nchunks - 1; c >= 0; --c)
        if (sh.cmass[c] > 0.f) {
          cs = c;
          before = __fsub_rn(W, sh.cmass[c]);
          break;
        }
    sh.ival[0] = (W > 0.f) ? cs : -1;
    sh.scal[1] = __fsub_rn(target, before);
    sh.scal[2] = W;
  }
  group_sync<kThreads>();
}

// Draw by the chunk masses in sh.cmass, then one pass over that chunk.  -1 when
// the masses sum to zero.  When the chunk's own running weight falls short of
// the located target (the masses were rounded differently), its last index
// with positive weight is taken.
template <class E, class WF>
SSD_DEV int chunked_draw(const VocabArgs &a, const char *rowT, const char *rowD, float u, const WF &wf,
                         float *W_out, Smem &sh) {
  locate_chunk(a.nchunks, u, sh);
  const int cs = sh.ival[0];
  const float local = sh.scal[1];
  *W_out = sh.scal[2];
  group_sync<kThreads>();
  if (cs < 0) return -1;
  const int start = cs * a.chunk_elems, end = min(a.V, start + a.chunk_elems);
  int d = range_find<E>(rowT, rowD, start, end, local, wf, sh);
  if (d < 0) {
    int last;
    (void)range_total<E>(rowT, rowD, start, end, wf, &last, sh);
    d = last;
  }
  return d;
}

// Exact chunk masses by one pass over every chunk of the row (used for Saguaro
// sampling when the down-weighted mass makes the statistics' masses inexact).
template <class E, class WF>
SSD_DEV void exact_chunk_masses(const VocabArgs &a, const char *rowT, const char *rowD, const WF &wf,
                                Smem &sh) {
  for (int c = 0; c < a.nchunks; ++c) {
    int last;
    const float t = range_total<E>(rowT, rowD, c * a.chunk_elems, min(a.V, (c + 1) * a.chunk_elems), wf, &last, sh);
    if (threadIdx.x == 0) sh.cmass[c] = t;
  }
  group_sync<kThreads>();
}

SSD_DEV float norm_N(float C, float sq) { return __fsub_rn(1.f, __fmul_rn(__fsub_rn(1.f, C), sq)); }

// Acceptance chain of sequence b: PosInfo and uniforms staged in shared memory
// by K threads, walked by thread 0.  Every thread returns the accept count.
SSD_DEV int chain(const VocabArgs &a, int b, Smem &sh) {
  for (int t = threadIdx.x; t < a.K; t += kThreads) {
    const PosInfo pi = a.pos[static_cast<size_t>(b) * a.K + t];
    sh.cp[t] = pi.p;
    sh.cq[t] = pi.q;
    sh.cu[t] = a.u_acc[static_cast<size_t>(b) * a.K + t];
  }
  group_sync<kThreads>();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int t = 0; t < a.K; ++t) {
      if (sh.cp[t] >= 0.f && __fmul_rn(sh.cu[t], sh.cq[t]) < sh.cp[t]) ++acc;
      else break;
    }
    sh.ival[1] = acc;
  }
  group_sync<kThreads>();
  const int acc = sh.ival[1];
  group_sync<kThreads>();
  return acc;
}

// ===========================================================================
// ROW item: merge row r, sample d_{r+1}, gather p(d), q'(d), write guesses
// ===========================================================================
template <class E>
__device__ __noinline__ void row_item(const VocabArgs &a, int b, int r, uint64_t *lists, Smem &sh) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int F = a.F[r];
  uint64_t *S = a.S + (static_cast<size_t>(b) * (a.K + 1) + r) * a.Fcap;
  // stage the chunk records of (target row r, draft row r) and the draft's candidate lists
  for (int c = tid; c < a.nchunks; c += kThreads) {
    if (a.tslot0 >= 0) sh.cs[0][c] = a.stats[chunk_index(a, b, a.tslot0 + r, c)];
    sh.cs[1][c] = a.stats[chunk_index(a, b, a.dslot0 + r, c)];
  }
  const bool lists_smem = a.nchunks * F <= kCandCap;
  if (lists_smem) {
    const uint64_t *src = a.cands + chunk_index(a, b, a.dslot0 + r, 0) * a.Fcap;
    for (int i = tid; i < a.nchunks * F; i += kThreads) lists[i] = src[(i / F) * a.Fcap + (i % F)];
  }
  group_sync<kThreads>();
  if (tid == 0) {
    RowInfo ri;
    memset(&ri, 0, sizeof(ri));
    if (a.tslot0 >= 0) {
      const RowStat t = merge_row_smem(a, sh.cs[0]);
      ri.mt = t.m;
      ri.st = t.s;
      ri.at = t.amax;
    }
    const RowStat d = merge_row_smem(a, sh.cs[1]);
    ri.md = d.m;
    ri.sd = d.s;
    ri.ad = d.amax;
    sh.ri = ri;
  }
  if (warp == 1) {
    if (lists_smem) merge_topf(lists, F, a.nchunks, F, sh.S);
    else merge_topf(a.cands + chunk_index(a, b, a.dslot0 + r, 0) * a.Fcap, a.Fcap, a.nchunks, F, sh.S);
  }
  group_sync<kThreads>();
  for (int i = tid; i < F; i += kThreads) S[i] = sh.S[i];  // for the residual and lookup items
  const float mdk = __fmul_rn(sh.ri.md, a.kT);
  if (tid == 0) {
    float sq = 0.f;
    if (!a.greedy && sh.ri.md != NEG_INF) {
      for (int i = 0; i < F; ++i)
        if (sh.S[i]) sq = __fadd_rn(sq, ex2(__fmaf_rn(cand_val(sh.S[i]), a.kT, -mdk)));
      sq = __fdiv_rn(sq, sh.ri.sd);
    }
    sh.ri.sq = sq;
  }
  group_sync<kThreads>();
  const RowInfo ri = sh.ri;
  const uint64_t keyF = F > 0 ? sh.S[F - 1] : 0ull;
  if (a.do_predict) {
    const int sumF = a.foff[a.K + 1];
    for (int i = tid; i < F; i += kThreads) {
      const uint64_t key = sh.S[i];
      a.guess[static_cast<size_t>(b) * sumF + a.foff[r] + i] = cand_idx(key);
      if (a.guess_q) {
        float q;
        if (a.greedy) q = (i == 0) ? 1.f : 0.f;
        else q = __fdiv_rn(ex2(__fmaf_rn(cand_val(key), a.kT, -mdk)), ri.sd);
        a.guess_q[static_cast<size_t>(b) * sumF + a.foff[r] + i] = q;
      }
    }
  }
  const char *rowD = row_ptr(a, 1, b, r, E::kSize);
  if (r < a.K && (a.do_sample || a.do_verify)) {
    int d;
    if (a.do_sample) {
      float qd;
      if (a.greedy) {
        d = ri.ad;
        qd = 1.f;
      } else {
        const WSaguaro wf{mdk, a.kT, a.C, keyF, F > 0};
        const float u = a.u_draft[static_cast<size_t>(b) * a.K + r];
        if (__fmul_rn(__fsub_rn(1.f, a.C), ri.sq) > 0.875f) {
          exact_chunk_masses<E>(a, nullptr, rowD, wf, sh);
        } else {
          // chunk masses of q' (unnormalised): s_c 2^(Mk_c - mdk) - (1 - C) sum_{i in S, in c} e_i
          for (int c = tid; c < a.nchunks; c += kThreads) {
            const ChunkStat cs = sh.cs[1][c];
            sh.cmass[c] = (cs.m == NEG_INF) ? 0.f : __fmul_rn(cs.s, ex2(__fsub_rn(__fmul_rn(cs.m, a.kT), mdk)));
          }
          group_sync<kThreads>();
          if (tid == 0 && a.C < 1.f) {
            for (int i = 0; i < F; ++i) {
              if (!sh.S[i]) continue;
              const int c = cand_idx(sh.S[i]) / a.chunk_elems;
              const float e = ex2(__fmaf_rn(cand_val(sh.S[i]), a.kT, -mdk));
              sh.cmass[c] = __fsub_rn(sh.cmass[c], __fmul_rn(__fsub_rn(1.f, a.C), e));
            }
            for (int c = 0; c < a.nchunks; ++c) sh.cmass[c] = fmaxf(sh.cmass[c], 0.f);
          }
          group_sync<kThreads>();
        }
        float W;
        d = chunked_draw<E>(a, nullptr, rowD, u, wf, &W, sh);
        if (d < 0) d = ri.ad;
        const float zd = E::ld(rowD, d);
        const bool ins = F > 0 && cand_key(zd, d) >= keyF;
        const float q = __fdiv_rn(ex2(__fmaf_rn(zd, a.kT, -mdk)), ri.sd);
        qd = __fdiv_rn(ins ? __fmul_rn(q, a.C) : q, norm_N(a.C, ri.sq));
      }
      if (tid == 0) {
        a.d_out[static_cast<size_t>(b) * a.K + r] = d;
        if (a.qd_out) a.qd_out[static_cast<size_t>(b) * a.K + r] = qd;
      }
    } else {
      d = a.d_in[static_cast<size_t>(b) * a.K + r];
    }
    if (a.do_verify && tid == 0) {
      PosInfo pi{d, 0.f, 0.f, 0};
      if (d >= 0 && d < a.V) {
        const float zt = E::ld(row_ptr(a, 0, b, r, E::kSize), d);
        const float zd = E::ld(rowD, d);
        if (a.greedy) {
          pi.p = (d == ri.at) ? 1.f : 0.f;
          pi.q = (d == ri.ad) ? 1.f : 0.f;
        } else {
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
  if (tid == 0) a.rows[static_cast<size_t>(b) * (a.K + 1) + r] = ri;
  signal_done(row_done(a, b));
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
// RES item: acceptance chain, residual mass of chunk c of row a
// ===========================================================================
template <class E>
__device__ __noinline__ void res_item(const VocabArgs &a, int b, int c, Smem &sh) {
  const int acc = chain(a, b, sh);
  ResInfo ri{0.f, -1};
  if (acc < a.K && !a.greedy) {
    const RowInfo row = a.rows[static_cast<size_t>(b) * (a.K + 1) + acc];
    const int F = a.F[acc];
    const uint64_t keyF = F > 0 ? a.S[(static_cast<size_t>(b) * (a.K + 1) + acc) * a.Fcap + F - 1] : 0ull;
    const WResidual wf = residual_weights(a, row, keyF, F);
    const int start = c * a.chunk_elems, end = min(a.V, start + a.chunk_elems);
    int last;
    ri.w = range_total<E>(row_ptr(a, 0, b, acc, E::kSize), row_ptr(a, 1, b, acc, E::kSize), start, end, wf,
                          &last, sh);
    ri.last = last;
  }
  if (threadIdx.x == 0) a.res[static_cast<size_t>(b) * a.nchunks + c] = ri;
  signal_done(res_done(a, b));
}

// ===========================================================================
// FIN item: bonus draw, outputs, cache lookup
// ===========================================================================
template <class E>
__device__ __noinline__ void fin_item(const VocabArgs &a, int b, Smem &sh) {
  const int tid = threadIdx.x;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int acc = chain(a, b, sh);
  const RowInfo row = a.rows[static_cast<size_t>(b) * (a.K + 1) + acc];
  const uint64_t *S = a.S + (static_cast<size_t>(b) * (a.K + 1) + acc) * a.Fcap;
  const int Fa = a.F[acc];
  const char *rowT = row_ptr(a, 0, b, acc, E::kSize);
  const char *rowD = row_ptr(a, 1, b, acc, E::kSize);
  const float ub = a.u_bonus[b];
  int bt = row.at;
  float W = 1.f;
  bool zero = false, draw_p = false;
  if (a.greedy) {
    if (acc < a.K) {
      W = (row.at != row.ad) ? 1.f : 0.f;
      zero = !(W > 0.f);
    }
  } else if (acc < a.K) {
    const ResInfo *res = a.res + static_cast<size_t>(b) * a.nchunks;
    for (int c = tid; c < a.nchunks; c += kThreads) sh.cmass[c] = res[c].w;
    group_sync<kThreads>();
    const WResidual wf = residual_weights(a, row, Fa > 0 ? S[Fa - 1] : 0ull, Fa);
    const int d = chunked_draw<E>(a, rowT, rowD, ub, wf, &W, sh);
    if (d >= 0) {
      bt = d;
    } else {
      zero = true;
      draw_p = true;
    }
  } else {
    draw_p = true;
  }
  if (draw_p && !a.greedy) {
    // p_{acc+1} drawn by its chunk masses from the statistics pass
    const float mtk = __fmul_rn(row.mt, a.kT);
    for (int c = tid; c < a.nchunks; c += kThreads) {
      const ChunkStat cs = a.stats[chunk_index(a, b, a.tslot0 + acc, c)];
      sh.cmass[c] = (cs.m == NEG_INF) ? 0.f : __fmul_rn(cs.s, ex2(__fsub_rn(__fmul_rn(cs.m, a.kT), mtk)));
    }
    group_sync<kThreads>();
    const WTarget wp{mtk, a.kT};
    float Wp;
    const int d = chunked_draw<E>(a, rowT, nullptr, ub, wp, &Wp, sh);
    bt = (d >= 0) ? d : row.at;
  }
  // lookup: the bonus among the F_a guesses of depth a
  if (a.do_lookup) {
    if (tid == 0) sh.ival[3] = 0x7fffffff;
    group_sync<kThreads>();
    for (int i = tid; i < Fa; i += kThreads)
      if (cand_idx(S[i]) == bt) atomicMin(&sh.ival[3], i);
    group_sync<kThreads>();
  }
  const int s_hit = (a.do_lookup && sh.ival[3] != 0x7fffffff) ? a.foff[acc] + sh.ival[3] : -1;
  // outputs, one element per thread
  if (tid <= a.K) {
    int v = -1;
    if (tid < acc) v = a.pos[static_cast<size_t>(b) * a.K + tid].d;
    if (tid == acc) v = bt;
    a.out_tokens[static_cast<size_t>(b) * (a.K + 1) + tid] = v;
  }
  if (a.do_lookup && a.next_tokens && tid < a.K)
    a.next_tokens[static_cast<size_t>(b) * a.K + tid] =
        (s_hit >= 0 && a.payload) ? a.payload[(static_cast<size_t>(b) * a.foff[a.K + 1] + s_hit) * a.K + tid] : -1;
  group_sync<kThreads>();
  if (tid == 0) {
    if (zero) atomicOr(a.status, kFlagZeroResidual);
    a.accept_len[b] = acc;
    a.bonus[b] = bt;
    if (a.resid_mass) a.resid_mass[b] = W;
    if (a.do_lookup) {
      if (a.slot_out) a.slot_out[b] = s_hit;
      if (s_hit >= 0) atomicAdd(a.ctr + 3, 1u);
    }
    __threadfence();
    const uint32_t done = atomicAdd(a.ctr + 2, 1u);
    if (done + 1 == static_cast<uint32_t>(a.B) && a.hits) {
      __threadfence();
      *a.hits = ld_acquire(a.ctr + 3);
    }
  }
  group_sync<kThreads>();
}

// ===========================================================================
// the persistent kernel
// ===========================================================================
SSD_DEV unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
SSD_DEV uint32_t ld_relaxed(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
SSD_DEV void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Work tickets passed from the scheduler warp to the compute warps.
constexpr int kTickets = 4;
struct Ticket {
  int kind, b, idx, stage;
  long q;  // queue position (trace)
};
struct Ring {
  Ticket t[kTickets];
  uint64_t tfull[kTickets], tempty[kTickets];  // ticket written / consumed
  uint64_t full[kStages], sempty[kStages];     // chunk landed / stage released
};

SSD_DEV bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Are the inputs of finish item f complete?  (Acquire: what its producers
// published is visible to this CTA once the ticket is handed over.)
SSD_DEV bool finish_ready(const VocabArgs &a, long f, Ticket &t) {
  int kind, b, idx;
  sched_decode(a.fs, f, kind, b, idx);
  const uint32_t *dep;
  uint32_t need;
  if (kind == IT_ROW) {
    dep = stats_done(a, b);
    need = a.fs.ns;
  } else if (kind == IT_RES) {
    dep = row_done(a, b);
    need = a.fs.nr;
  } else {
    dep = res_done(a, b);
    need = a.fs.nc;
  }
  t.kind = kind;
  t.b = b;
  t.idx = idx;
  t.stage = -1;
  t.q = a.nst + f;
  return ld_acquire(dep) >= need;
}

// The scheduler warp's lane 0.  Work is assigned round robin over the grid:
// statistics chunk q to CTA q mod G, finish item f to CTA f mod G.  Each pass
// it (1) keeps the copy ring full -- a chunk copy is issued as soon as a stage
// and a ticket slot are free (non-blocking tests) -- and (2) hands over any of
// its pending finish items whose inputs are complete, in any order.  No item
// waits once handed over, so nothing can deadlock on the compute side; the
// pending finish items of this CTA only wait for other CTAs' published work.
constexpr int kWindow = 64;  // pending finish items scanned per pass
constexpr int kChecksPerPass = 4;
template <class E>
SSD_DEV void scheduler(const VocabArgs &a, uint8_t *buf, Ring &R) {
  const long G = gridDim.x;
  const long fin_total = sched_total(a.fs);
  const long my_stats = (a.nst > blockIdx.x) ? (a.nst - blockIdx.x + G - 1) / G : 0;
  const long my_fin = (fin_total > blockIdx.x) ? (fin_total - blockIdx.x + G - 1) / G : 0;
  long k = 0;       // statistics chunks issued
  long w = 0;       // tickets written
  long j_lo = 0;    // finish items below j_lo are all handed over
  uint64_t done_mask = 0;  // handed-over items in [j_lo, j_lo + 64)
  long fin_left = my_fin;
  uint32_t idle = 0;
  for (;;) {
    bool progress = false;
    // (1) statistics copies
    while (k < my_stats) {
      const int slot = static_cast<int>(w % kTickets);
      if (w >= kTickets && !mbar_test(&R.tempty[slot], static_cast<uint32_t>((w / kTickets - 1) & 1))) break;
      const int st = static_cast<int>(k % kStages);
      if (k >= kStages && !mbar_test(&R.sempty[st], static_cast<uint32_t>((k / kStages - 1) & 1))) break;
      const long q = blockIdx.x + k * G;
      Ticket t;
      t.kind = IT_STATS;
      t.b = static_cast<int>(q / a.fs.ns);
      t.idx = static_cast<int>(q % a.fs.ns);
      t.stage = st;
      t.q = q;
      fence_proxy_async();
      issue_stats<E>(a, t.b, t.idx, buf + st * kChunkBytes, &R.full[st]);
      R.t[slot] = t;
      mbar_arrive(&R.tfull[slot]);
      ++w;
      ++k;
      progress = true;
    }
    // (2) finish items whose inputs are complete
    int checks = 0;
    for (int jj = 0; jj < kWindow && fin_left > 0 && checks < kChecksPerPass; ++jj) {
      const long j = j_lo + jj;
      const long f = blockIdx.x + j * G;
      if (f >= fin_total) break;
      if ((done_mask >> jj) & 1ull) continue;
      const int slot = static_cast<int>(w % kTickets);
      if (w >= kTickets && !mbar_test(&R.tempty[slot], static_cast<uint32_t>((w / kTickets - 1) & 1))) break;
      Ticket t;
      ++checks;
      if (!finish_ready(a, f, t)) continue;
      R.t[slot] = t;
      mbar_arrive(&R.tfull[slot]);
      ++w;
      --fin_left;
      done_mask |= 1ull << jj;
      progress = true;
    }
    while (done_mask & 1ull) {  // slide the window past a handed-over prefix
      done_mask >>= 1;
      ++j_lo;
    }
    if (k == my_stats && fin_left == 0) break;
    if (!progress) {
      if (ld_relaxed(a.ctr + 1) != 0 || ++idle > kMaxSpins) {
        atomicOr(a.status, kFlagWaitTimeout);
        atomicExch(a.ctr + 1, 1u);
        break;
      }
      __nanosleep(64);
    } else {
      idle = 0;
    }
  }
  // end of work for the compute warps
  const int slot = static_cast<int>(w % kTickets);
  if (w >= kTickets) (void)mbar_wait(&R.tempty[slot], static_cast<uint32_t>((w / kTickets - 1) & 1));
  R.t[slot].kind = IT_NONE;
  mbar_arrive(&R.tfull[slot]);
}

template <class E>
__global__ void __maxnreg__(112) k_vocab(const VocabArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *buf = smem;
  uint64_t *cand = reinterpret_cast<uint64_t *>(smem + kStages * kChunkBytes);
  Smem &sh = *reinterpret_cast<Smem *>(smem + kStages * kChunkBytes + kCandCap * sizeof(uint64_t));
  __shared__ __align__(8) Ring R;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kTickets; ++i) {
      mbar_init(&R.tfull[i], 1);
      mbar_init(&R.tempty[i], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&R.full[s], 1);
      mbar_init(&R.sempty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid >= kThreads) {
    if (tid == kThreads) scheduler<E>(a, buf, R);
    return;
  }
  // compute warps: take tickets in order
  long r = 0;
  for (;;) {
    const int slot = static_cast<int>(r % kTickets);
    const bool got = mbar_wait(&R.tfull[slot], static_cast<uint32_t>((r / kTickets) & 1));
    if (group_sync_or<kThreads>(!got)) {
      if (tid == 0) {
        atomicOr(a.status, kFlagWaitTimeout);
        atomicExch(a.ctr + 1, 1u);
      }
      break;
    }
    const Ticket t = R.t[slot];
    if (t.kind == IT_NONE) break;
    const unsigned long long t0 = (a.trace && tid == 0) ? globaltimer() : 0ull;
    if (t.kind == IT_STATS) {
      const long n = t.q / gridDim.x;  // this CTA's ordinal of the item
      const bool ok = mbar_wait(&R.full[t.stage], static_cast<uint32_t>((n / kStages) & 1));
      if (group_sync_or<kThreads>(!ok)) {
        if (tid == 0) {
          atomicOr(a.status, kFlagWaitTimeout);
          atomicExch(a.ctr + 1, 1u);
        }
        // the copy may still land: a last bounded wait before leaving
        if (tid == 0) (void)mbar_wait(&R.full[t.stage], static_cast<uint32_t>((n / kStages) & 1));
        break;
      }
      stats_item<E>(a, t.b, t.idx, buf + t.stage * kChunkBytes, cand, sh);
      if (tid == 0) mbar_arrive(&R.sempty[t.stage]);
    } else if (t.kind == IT_ROW) {
      row_item<E>(a, t.b, t.idx, cand, sh);
    } else if (t.kind == IT_RES) {
      res_item<E>(a, t.b, t.idx, sh);
    } else {
      fin_item<E>(a, t.b, sh);
    }
    group_sync<kThreads>();
    if (tid == 0) {
      mbar_arrive(&R.tempty[slot]);
      if (a.trace) {
        unsigned long long *tr = a.trace + 4 * t.q;
        tr[0] = (static_cast<unsigned long long>(blockIdx.x) << 48) |
                (static_cast<unsigned long long>(t.kind) << 40) | (static_cast<unsigned long long>(t.b) << 20) |
                static_cast<unsigned long long>(t.idx);
        tr[1] = t0;
        tr[2] = t0;
        tr[3] = globaltimer();
      }
    }
    ++r;
  }
}

// Cache lookup alone (one CTA; hits written, not accumulated).
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
  group_sync<kThreads>();
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
  group_sync<kThreads>();
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
  size_t ctr_off, stats_off, cands_off, rows_off, S_off, pos_off, res_off, total;
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
  size_t o = 0;
  L->ctr_off = o;
  o = align_up(o + (4 + 3 * Bn) * sizeof(uint32_t), 256);
  L->stats_off = o;
  o = align_up(o + nrec * sizeof(ChunkStat), 256);
  L->cands_off = o;
  o = align_up(o + nrec * L->Fcap * sizeof(uint64_t), 256);
  L->rows_off = o;
  o = align_up(o + Bn * (K + 1) * sizeof(RowInfo), 256);
  L->S_off = o;
  o = align_up(o + Bn * (K + 1) * L->Fcap * sizeof(uint64_t), 256);
  L->pos_off = o;
  o = align_up(o + Bn * (K > 0 ? K : 1) * sizeof(PosInfo), 256);
  L->res_off = o;
  o = align_up(o + Bn * L->nchunks * sizeof(ResInfo), 256);
  L->total = o;
  return true;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
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
  a.cands = reinterpret_cast<uint64_t *>(w + L.cands_off);
  a.rows = reinterpret_cast<RowInfo *>(w + L.rows_off);
  a.S = reinterpret_cast<uint64_t *>(w + L.S_off);
  a.pos = reinterpret_cast<PosInfo *>(w + L.pos_off);
  a.res = reinterpret_cast<ResInfo *>(w + L.res_off);
  a.status = status;
  a.tslot0 = -1;
  return a;
}

void set_slots(VocabArgs &a, bool target_rows, int ndraft) {
  int n = 0;
  if (target_rows) {
    a.tslot0 = 0;
    for (int r = 0; r <= a.K; ++r) a.slot[n++] = RowSlot{0, static_cast<int16_t>(r), 0, 0};
  }
  a.dslot0 = n;
  for (int r = 0; r < ndraft; ++r)
    a.slot[n++] = RowSlot{1, static_cast<int16_t>(r), static_cast<int16_t>(a.F[r]), 0};
  a.nslots = n;
}

// Optional timing hook (ssd_set_timing_events): events recorded around the
// persistent kernel of every vocabulary call while set.
cudaEvent_t g_ev_before = nullptr;
cudaEvent_t g_ev_after = nullptr;
// Optional per-entry trace (ssd_set_trace).
void *g_trace = nullptr;
size_t g_trace_bytes = 0;

constexpr size_t kVocabSmem = kStages * kChunkBytes + kCandCap * sizeof(uint64_t) + sizeof(Smem);
// two resident CTAs per SM: 2 x (dynamic + static + 1 KiB reserved) <= 228 KiB
static_assert(2 * (kVocabSmem + 1024 + 512) <= 228 * 1024, "shared memory of k_vocab too large for 2 CTAs/SM");

template <class E>
cudaError_t launch_vocab(VocabArgs &a, int nr, int nc, int nf, cudaStream_t s) {
  constexpr int kBlock = kThreads + 32;  // 8 compute warps + the scheduler warp
  cudaError_t e = cudaFuncSetAttribute(k_vocab<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kVocabSmem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_vocab<E>, kBlock, kVocabSmem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  Sched fs;
  fs.B = a.B;
  fs.ns = a.nslots * a.nchunks;
  fs.nr = nr;
  fs.nc = nc;
  fs.nf = nf;
  fs.L1 = 0;
  fs.L2 = 1;
  fs.L3 = 2;
  a.fs = fs;
  a.nst = static_cast<long>(a.B) * fs.ns;
  const long fin_total = sched_total(fs);
  long grid = static_cast<long>(num_sms()) * per_sm;
  if (grid > a.nst + fin_total) grid = a.nst + fin_total;
  if (grid < 1) return cudaSuccess;
  a.trace = (g_trace && g_trace_bytes >= static_cast<size_t>(a.nst + fin_total) * 32)
                ? static_cast<unsigned long long *>(g_trace)
                : nullptr;
  // the finish-queue head, abort flag, counters start at zero
  e = cudaMemsetAsync(a.ctr, 0, (4 + 3 * static_cast<size_t>(a.B)) * sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  if (g_ev_before) cudaEventRecord(g_ev_before, s);
  k_vocab<E><<<static_cast<unsigned>(grid), kBlock, kVocabSmem, s>>>(a);
  e = cudaGetLastError();
  if (g_ev_after) cudaEventRecord(g_ev_after, s);
  return e;
}

cudaError_t launch_any(ssd_dtype_t dt, VocabArgs &a, int nr, int nc, int nf, cudaStream_t s) {
  return dt == SSD_F32 ? launch_vocab<EF32>(a, nr, nc, nf, s) : launch_vocab<EBF16>(a, nr, nc, nf, s);
}

ssd_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

// Fixed device scratch for ssd_verify_noalloc: one array per GPU that loads
// the library, held until the process exits.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
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
  set_slots(a, false, K);
  a.do_sample = 1;
  a.u_draft = u_draft;
  a.d_out = d_out;
  a.qd_out = qd_out;
  return cuda_status(launch_any(dt, a, K, 0, 0, reinterpret_cast<cudaStream_t>(s)));
}

ssd_status_t ssd_verify(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                        int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                        const int32_t *d, const float *u_acc, const float *u_bonus, int32_t *accept_len,
                        int32_t *out_tokens, int32_t *bonus, float *accept_prob, float *resid_mass,
                        uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s) {
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
  set_slots(a, true, K + 1);
  a.do_verify = 1;
  a.d_in = d;
  a.u_acc = u_acc;
  a.u_bonus = u_bonus;
  a.accept_len = accept_len;
  a.out_tokens = out_tokens;
  a.bonus = bonus;
  a.accept_prob = accept_prob;
  a.resid_mass = resid_mass;
  return cuda_status(launch_any(dt, a, K + 1, L.nchunks, 1, reinterpret_cast<cudaStream_t>(s)));
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
  set_slots(a, false, K + 1);
  a.do_predict = 1;
  a.guess = guess;
  a.guess_q = guess_q;
  return cuda_status(launch_any(dt, a, K + 1, 0, 0, reinterpret_cast<cudaStream_t>(s)));
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
                       int32_t *next_tokens, uint32_t *hits, uint32_t *status, void *ws, size_t ws_bytes,
                       ssd_stream_t s) {
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
  set_slots(a, true, K + 1);
  a.do_sample = 1;
  a.do_verify = 1;
  a.do_predict = guess != nullptr;
  a.do_lookup = guess != nullptr;
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
  return cuda_status(launch_any(dt, a, K + 1, L.nchunks, 1, cs));
}

size_t ssd_verify_noalloc_max_bytes(void) { return kStaticScratchBytes; }

ssd_status_t ssd_verify_noalloc(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                                int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                                const int32_t *d, const float *u_acc, const float *u_bonus,
                                int32_t *accept_len, int32_t *out_tokens, int32_t *bonus, float *accept_prob,
                                float *resid_mass, uint32_t *status, ssd_stream_t s) {
  Layout L;
  if (!F || !make_layout(B, K, V, dt, F, &L))
    return (F && B >= 0 && K >= 0 && V >= 1) ? SSD_ERR_UNSUPPORTED : SSD_ERR_INVALID_ARG;
  if (L.total > kStaticScratchBytes) return SSD_ERR_WORKSPACE;  // the batch needs more scratch than the array holds
  if (B == 0) return ssd_verify(target, draft, dt, seq_stride, row_stride, B, K, V, F, C, T, d, u_acc, u_bonus,
                                accept_len, out_tokens, bonus, accept_prob, resid_mass, status, nullptr, 0, s);
  void *ws = nullptr;
  if (static_scratch(&ws) != cudaSuccess) return SSD_ERR_CUDA;
  return ssd_verify(target, draft, dt, seq_stride, row_stride, B, K, V, F, C, T, d, u_acc, u_bonus, accept_len,
                    out_tokens, bonus, accept_prob, resid_mass, status, ws, kStaticScratchBytes, s);
}

}  // extern "C"
