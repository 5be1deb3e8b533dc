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
// Structure (all calls):
//   1. k_row_stats: one persistent, HBM-bound pass over every logit row the
//      call needs.  Each CTA owns a ring of two 32 KiB shared-memory stages
//      filled by TMA bulk copies (cp.async.bulk + mbarrier); per 32 KiB chunk
//      it produces (max, sum of 2^((z-max)/T*log2 e), argmax, top-F
//      candidates) into the workspace.  This pass moves >= 95% of the bytes.
//   2. small finish kernels merge the per-chunk records of a row (a k-way
//      merge of sorted candidate lists for top-F) and do the per-sequence
//      work: inverse-CDF draws, the acceptance chain, the residual draw,
//      guesses and the cache lookup.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/ssd.h"
#include "common.cuh"

namespace ssd {

constexpr int kStatsThreads = 256;
constexpr int kChunkBytes = 32768;
constexpr int kStages = 2;
constexpr int kCandCap = 1024;
constexpr int kMaxK = 16;
constexpr int kMaxSlots = 2 * (kMaxK + 1);
constexpr int kMaxF = 256;
constexpr int kMaxChunks = 128;  // per row: 4 lists per lane in the warp merge
constexpr int kFinishThreads = 256;
constexpr int kMaxTiles = 4096;  // inverse-CDF tiles per row

struct ChunkStat {
  float m;       // chunk maximum
  float s;       // sum of 2^((z - m) * kT) over the chunk (0 when greedy)
  float amax_v;  // == m
  int amax_i;    // lowest index holding m
};

struct RowSlot {
  int16_t tensor;  // 0 = target, 1 = draft
  int16_t row;     // row r (position r + 1)
  int16_t F;       // top-F candidates wanted (0 = none)
  int16_t pad;
};

struct VocabArgs {
  const void *target;
  const void *draft;
  int64_t seq_stride, row_stride;  // elements
  int B, K, V;
  int nslots, nchunks, chunk_elems, Fcap;
  float kT;    // log2(e) / T; unused when greedy
  int greedy;  // T == 0
  float C;
  RowSlot slot[kMaxSlots];
  int F[kMaxK + 1];
  int foff[kMaxK + 2];  // prefix sums of F
  ChunkStat *stats;     // [B][nslots][nchunks]
  uint64_t *cands;      // [B][nslots][nchunks][Fcap]
  uint32_t *status;
};

__host__ __device__ inline size_t chunk_index(const VocabArgs &a, int b, int slot, int c) {
  return (static_cast<size_t>(b) * a.nslots + slot) * a.nchunks + c;
}

SSD_DEV const char *row_ptr(const VocabArgs &a, int tensor, int b, int row, int esize) {
  const char *base = reinterpret_cast<const char *>(tensor ? a.draft : a.target);
  return base + (static_cast<int64_t>(b) * a.seq_stride + static_cast<int64_t>(row) * a.row_stride) * esize;
}

// ===========================================================================
// 1. row statistics
// ===========================================================================
template <class E>
SSD_DEV void issue_chunk(const VocabArgs &a, long item, uint8_t *dst, uint64_t *bar) {
  const int c = static_cast<int>(item % a.nchunks);
  const long rest = item / a.nchunks;
  const int slot = static_cast<int>(rest % a.nslots);
  const int b = static_cast<int>(rest / a.nslots);
  const RowSlot rs = a.slot[slot];
  const int e0 = c * a.chunk_elems;
  const int n = min(a.chunk_elems, a.V - e0);
  const uint32_t bulk = static_cast<uint32_t>((n * E::kSize) & ~15);
  const char *src = row_ptr(a, rs.tensor, b, rs.row, E::kSize) + static_cast<int64_t>(e0) * E::kSize;
  mbar_arrive_expect_tx(bar, bulk);
  if (bulk) bulk_g2s(dst, src, bulk, bar);
}

struct StatsShared {
  float red[32];
  uint64_t redk[32];
  int amax;
  int ncand;
};

// Per-chunk statistics of `item` from the staged bytes in `buf`.
template <class E>
SSD_DEV void chunk_stats(const VocabArgs &a, long item, const uint8_t *buf, uint64_t *cand,
                         StatsShared &sh) {
  constexpr int NT = kStatsThreads;
  const int tid = threadIdx.x;
  const int c = static_cast<int>(item % a.nchunks);
  const long rest = item / a.nchunks;
  const int slot = static_cast<int>(rest % a.nslots);
  const int b = static_cast<int>(rest / a.nslots);
  const RowSlot rs = a.slot[slot];
  const int e0 = c * a.chunk_elems;
  const int n = min(a.chunk_elems, a.V - e0);
  const int nvec = (n * E::kSize) >> 4;
  const int nbulk = nvec * E::kVec;
  const int ntail = n - nbulk;
  const char *row = row_ptr(a, rs.tensor, b, rs.row, E::kSize);
  const uint4 *v4 = reinterpret_cast<const uint4 *>(buf);
  const float kT = a.kT;
  const bool greedy = a.greedy != 0;
  const float NEG_INF = -__int_as_float(0x7f800000);

  // ---- streaming pass: running max and rescaled sum of 2^((z - m) kT)
  float m = NEG_INF, s = 0.f;
  int cnt = 0;
  for (int v = tid; v < nvec; v += NT) {
    float f[E::kVec];
    E::unpack(v4[v], f);
    float vm = f[0];
#pragma unroll
    for (int e = 1; e < E::kVec; ++e) vm = fmaxf(vm, f[e]);
    if (vm > m) {
      if (!greedy && m != NEG_INF) s = __fmul_rn(s, ex2(__fmul_rn(__fsub_rn(m, vm), kT)));
      m = vm;
    }
    if (!greedy && m != NEG_INF) {
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) s = __fadd_rn(s, ex2(__fmul_rn(__fsub_rn(f[e], m), kT)));
    }
    ++cnt;
  }
  float zt = NEG_INF;
  if (tid < ntail) {
    zt = E::ld(row, e0 + nbulk + tid);
    if (zt > m) {
      if (!greedy && m != NEG_INF) s = __fmul_rn(s, ex2(__fmul_rn(__fsub_rn(m, zt), kT)));
      m = zt;
    }
    if (!greedy && m != NEG_INF) s = __fadd_rn(s, ex2(__fmul_rn(__fsub_rn(zt, m), kT)));
    ++cnt;
  }

  // ---- chunk max and sum
  const float M = block_max<NT>(m, sh.red);
  float sr = 0.f;
  if (!greedy && m != NEG_INF) sr = __fmul_rn(s, ex2(__fmul_rn(__fsub_rn(m, M), kT)));
  const float S = greedy ? 0.f : block_sum<NT>(sr, sh.red);

  // ---- argmax: only threads holding the maximum rescan their elements
  if (tid == 0) sh.amax = 0x7fffffff;
  __syncthreads();
  if (cnt > 0 && m == M) {
    int best = 0x7fffffff;
    for (int v = tid; v < nvec && best == 0x7fffffff; v += NT) {
      float f[E::kVec];
      E::unpack(v4[v], f);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e)
        if (f[e] == M && best == 0x7fffffff) best = v * E::kVec + e;
    }
    if (best == 0x7fffffff && tid < ntail && zt == M) best = nbulk + tid;
    atomicMin(&sh.amax, best);
  }
  __syncthreads();
  const int amax = e0 + sh.amax;

  // ---- top-F candidates of the chunk
  const int F = rs.F;
  uint64_t *out = a.cands + chunk_index(a, b, slot, c) * a.Fcap;
  if (F == 1) {
    if (tid == 0) out[0] = cand_key(M, amax);
  } else if (F > 1) {
    // threshold tau: the F-th largest per-thread maximum (keys of empty threads are 0);
    // at least F elements of the chunk have key >= tau.
    const uint32_t mykey = cnt ? f2ord(m) : 0u;
    uint32_t tau = 0;
    for (int bit = 31; bit >= E::kLowBit; --bit) {
      const uint32_t t = tau | (1u << bit);
      if (__syncthreads_count(mykey >= t) >= F) tau = t;
    }
    if (tid == 0) sh.ncand = 0;
    __syncthreads();
    if (cnt && mykey >= tau) {
      for (int v = tid; v < nvec; v += NT) {
        float f[E::kVec];
        E::unpack(v4[v], f);
#pragma unroll
        for (int e = 0; e < E::kVec; ++e)
          if (f2ord(f[e]) >= tau) {
            const int pos = atomicAdd(&sh.ncand, 1);
            if (pos < kCandCap) cand[pos] = cand_key(f[e], e0 + v * E::kVec + e);
          }
      }
      if (tid < ntail && f2ord(zt) >= tau) {
        const int pos = atomicAdd(&sh.ncand, 1);
        if (pos < kCandCap) cand[pos] = cand_key(zt, e0 + nbulk + tid);
      }
    }
    __syncthreads();
    const int nc = sh.ncand;
    if (nc <= kCandCap) {
      int P = 1;
      while (P < nc || P < F) P <<= 1;
      for (int i = nc + tid; i < P; i += NT) cand[i] = 0ull;
      __syncthreads();
      // bitonic sort, descending
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
          __syncthreads();
        }
      }
      for (int i = tid; i < F; i += NT) out[i] = cand[i];
    } else {
      // too many ties at the threshold: exact selection, one winner per sweep
      uint64_t prev = ~0ull;
      for (int r = 0; r < F; ++r) {
        uint64_t best = 0;
        for (int v = tid; v < nvec; v += NT) {
          float f[E::kVec];
          E::unpack(v4[v], f);
#pragma unroll
          for (int e = 0; e < E::kVec; ++e) {
            const uint64_t key = cand_key(f[e], e0 + v * E::kVec + e);
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
  }
  if (tid == 0) {
    ChunkStat cs;
    cs.m = M;
    cs.s = S;
    cs.amax_v = M;
    cs.amax_i = amax;
    a.stats[chunk_index(a, b, slot, c)] = cs;
  }
  __syncthreads();
}

template <class E>
__global__ void __launch_bounds__(kStatsThreads, 3) k_row_stats(const VocabArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *buf = smem;
  uint64_t *cand = reinterpret_cast<uint64_t *>(smem + kStages * kChunkBytes);
  __shared__ __align__(8) uint64_t bar[kStages];
  __shared__ StatsShared sh;
  const int tid = threadIdx.x;
  const long total = static_cast<long>(a.B) * a.nslots * a.nchunks;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      const long it = blockIdx.x + static_cast<long>(s) * gridDim.x;
      if (it < total) issue_chunk<E>(a, it, buf + s * kChunkBytes, &bar[s]);
    }
  }
  uint32_t phase = 0;
  int k = 0;
  bool timed_out = false;
  for (long it = blockIdx.x; it < total; it += gridDim.x, ++k) {
    const int st = k % kStages;
    const bool ok = mbar_wait(&bar[st], (phase >> st) & 1u);
    phase ^= 1u << st;
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    chunk_stats<E>(a, it, buf + st * kChunkBytes, cand, sh);
    const long nx = it + static_cast<long>(kStages) * gridDim.x;
    if (tid == 0 && nx < total) {
      fence_proxy_async();
      issue_chunk<E>(a, nx, buf + st * kChunkBytes, &bar[st]);
    }
  }
  if (timed_out && tid == 0) {
    atomicOr(a.status, kFlagWaitTimeout);
    // drain copies still in flight before the CTA's shared memory is released
    for (int s = 0; s < kStages; ++s) (void)mbar_wait(&bar[s], (phase >> s) & 1u);
  }
}

// ===========================================================================
// 2. per-row merge of the chunk records
// ===========================================================================
struct RowStat {
  float m, s;
  int amax;
};

SSD_DEV RowStat merge_row(const VocabArgs &a, int b, int slot) {
  // chunks are in index order, so a strictly larger maximum keeps the lowest index
  const float NEG_INF = -__int_as_float(0x7f800000);
  const ChunkStat c0 = a.stats[chunk_index(a, b, slot, 0)];
  RowStat r;
  r.m = c0.m;
  r.amax = c0.amax_i;
  for (int c = 1; c < a.nchunks; ++c) {
    const ChunkStat cs = a.stats[chunk_index(a, b, slot, c)];
    if (cs.m > r.m) {
      r.m = cs.m;
      r.amax = cs.amax_i;
    }
  }
  r.s = 0.f;
  if (!a.greedy && r.m != NEG_INF) {
    for (int c = 0; c < a.nchunks; ++c) {
      const ChunkStat cs = a.stats[chunk_index(a, b, slot, c)];
      if (cs.m != NEG_INF) r.s = __fadd_rn(r.s, __fmul_rn(cs.s, ex2(__fmul_rn(__fsub_rn(cs.m, r.m), a.kT))));
    }
  }
  return r;
}

// Warp-cooperative k-way merge of the sorted per-chunk candidate lists of one
// row into its top-F list (descending keys; sentinel 0 past the end).
SSD_DEV void merge_topf(const VocabArgs &a, int b, int slot, int F, uint64_t *dst) {
  constexpr int L = kMaxChunks / 32;
  const int lane = threadIdx.x & 31;
  int ptr[L];
  uint64_t head[L];
  const uint64_t *base = a.cands + chunk_index(a, b, slot, 0) * a.Fcap;
#pragma unroll
  for (int l = 0; l < L; ++l) {
    const int c = lane + 32 * l;
    ptr[l] = 0;
    head[l] = (c < a.nchunks && F > 0) ? base[static_cast<size_t>(c) * a.Fcap] : 0ull;
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
      // keys are unique (the index is part of the key), so one lane advances
#pragma unroll
      for (int l = 0; l < L; ++l)
        if (l == bl) {
          const int c = lane + 32 * l;
          ++ptr[l];
          head[l] = (ptr[l] < F) ? base[static_cast<size_t>(c) * a.Fcap + ptr[l]] : 0ull;
        }
    }
  }
  __syncwarp();
}

// ===========================================================================
// 3. inverse-CDF draw over one row (one CTA)
// ===========================================================================
struct InvCdfShared {
  float red[kFinishThreads / 32 + 1];
  float tile_tot[kMaxTiles];
  int last_pos;
  int found;
  int gstar;
  float cum_g, target, W;
};

// Weight functors: operator()(zt, zd, idx) -> weight >= 0, with a fixed
// sequence of correctly-rounded operations so that both passes agree bit for bit.
struct WSaguaro {  // unnormalised q'_i
  float md, kT, C;
  uint64_t keyF;
  bool hasS;
  SSD_DEV float operator()(float, float zd, int idx) const {
    const float e = ex2(__fmul_rn(__fsub_rn(zd, md), kT));
    return (hasS && cand_key(zd, idx) >= keyF) ? __fmul_rn(e, C) : e;
  }
};
struct WTarget {  // unnormalised p_i
  float mt, kT;
  SSD_DEV float operator()(float zt, float, int) const { return ex2(__fmul_rn(__fsub_rn(zt, mt), kT)); }
};
struct WResidual {  // max(0, p_i - q'_i)
  float mt, kT, inv_st, md, fC, f1;
  uint64_t keyF;
  bool hasS;
  SSD_DEV float operator()(float zt, float zd, int idx) const {
    const float p = __fmul_rn(ex2(__fmul_rn(__fsub_rn(zt, mt), kT)), inv_st);
    const float f = (hasS && cand_key(zd, idx) >= keyF) ? fC : f1;
    const float q = __fmul_rn(ex2(__fmul_rn(__fsub_rn(zd, md), kT)), f);
    const float r = __fsub_rn(p, q);
    return r > 0.f ? r : 0.f;
  }
};

template <class E, class WF>
SSD_DEV float tile_weights(const void *rowT, const void *rowD, int V, int i0, const WF &wf,
                           float *w, int *lastpos) {
  float fz[E::kVec], fd[E::kVec];
  bool vt[E::kVec], vd[E::kVec];
  if (rowT) load_vec<E>(rowT, i0, V, fz, vt);
  if (rowD) load_vec<E>(rowD, i0, V, fd, vd);
  float t = 0.f;
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) {
    const bool valid = (i0 + e) < V;
    const float x = valid ? wf(rowT ? fz[e] : 0.f, rowD ? fd[e] : 0.f, i0 + e) : 0.f;
    w[e] = x;
    t = __fadd_rn(t, x);
    if (x > 0.f) *lastpos = i0 + e;
  }
  return t;
}

// Smallest i with sum_{k<=i} w_k > u * W (W = sum of all w), or the last index
// with w > 0 when rounding leaves none; -1 when W <= 0.  All threads return
// the same value; *W_out receives W.
template <class E, class WF>
SSD_DEV int block_inv_cdf(const void *rowT, const void *rowD, int V, float u, const WF &wf,
                          float *W_out, InvCdfShared &sh) {
  constexpr int NT = kFinishThreads;
  constexpr int TILE = NT * E::kVec;
  const int tid = threadIdx.x;
  const int ntiles = (V + TILE - 1) / TILE;
  int lastpos = -1;
  float w[E::kVec];
  if (tid == 0) {
    sh.last_pos = -1;
    sh.found = 0x7fffffff;
  }
  for (int g = 0; g < ntiles; ++g) {
    const int i0 = g * TILE + tid * E::kVec;
    const float t = tile_weights<E>(rowT, rowD, V, i0, wf, w, &lastpos);
    const float ex = block_excl_scan<NT>(t, sh.red);
    if (tid == NT - 1) sh.tile_tot[g] = __fadd_rn(ex, t);
  }
  atomicMax(&sh.last_pos, lastpos);
  __syncthreads();
  if (tid == 0) {
    float cum = 0.f;
    for (int g = 0; g < ntiles; ++g) cum = __fadd_rn(cum, sh.tile_tot[g]);
    const float W = cum;
    const float target = __fmul_rn(u, W);
    int gs = -1;
    float cg = 0.f, c = 0.f;
    for (int g = 0; g < ntiles; ++g) {
      const float nc = __fadd_rn(c, sh.tile_tot[g]);
      if (nc > target) {
        gs = g;
        cg = c;
        break;
      }
      c = nc;
    }
    sh.W = W;
    sh.gstar = (W > 0.f) ? gs : -2;
    sh.cum_g = cg;
    sh.target = target;
  }
  __syncthreads();
  const int gs = sh.gstar;
  const int last = sh.last_pos;
  *W_out = sh.W;
  int result = (gs == -2) ? -1 : last;
  if (gs >= 0) {
    const int i0 = gs * TILE + tid * E::kVec;
    int dummy = -1;
    const float t = tile_weights<E>(rowT, rowD, V, i0, wf, w, &dummy);
    const float ex = block_excl_scan<NT>(t, sh.red);
    const float cg = sh.cum_g, target = sh.target;
    float run = 0.f;
    int hit = 0x7fffffff;
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) {
      run = __fadd_rn(run, w[e]);
      const float x = __fadd_rn(cg, __fadd_rn(ex, run));
      if (x > target && hit == 0x7fffffff && w[e] > 0.f) hit = i0 + e;
    }
    if (hit != 0x7fffffff) atomicMin(&sh.found, hit);
    __syncthreads();
    const int f = sh.found;
    if (f != 0x7fffffff) result = f;
  }
  // every thread has read the shared state before a later call may reset it
  __syncthreads();
  return result;
}

// ===========================================================================
// 4. finish kernels
// ===========================================================================
struct FinishOut {
  // sampling
  const float *u_draft;
  int32_t *d_out;
  float *qd_out;
  // verification
  const int32_t *d_in;
  const float *u_acc;
  const float *u_bonus;
  int32_t *accept_len, *out_tokens, *bonus;
  float *accept_prob, *resid_mass;
  // prediction + lookup
  int32_t *guess;
  float *guess_q;
  const int32_t *payload;
  int32_t *slot, *next_tokens;
  uint32_t *hits;
  int tslot0, dslot0;  // slot index of target row 0 and draft row 0
};

struct SeqShared {
  RowStat rs[kMaxSlots];
  float sq[kMaxK + 1];  // sum of q over S_j per draft row
  float p[kMaxK], qp[kMaxK];
  int acc_len;
  InvCdfShared inv;
};

// q'(i) factors of draft row r: c_i / (s * N)
SSD_DEV float norm_N(float C, float sq) { return __fsub_rn(1.f, __fmul_rn(__fsub_rn(1.f, C), sq)); }

// Saguaro sampling: one CTA per (position j, sequence b).
template <class E>
__global__ void __launch_bounds__(kFinishThreads) k_sample_finish(const VocabArgs a, const FinishOut o) {
  extern __shared__ __align__(16) uint8_t dsm[];
  uint64_t *S = reinterpret_cast<uint64_t *>(dsm);  // [Fcap]
  __shared__ RowStat rs;
  __shared__ InvCdfShared inv;
  __shared__ float s_sq;
  const int r = blockIdx.x, b = blockIdx.y;
  const int slot = o.dslot0 + r;
  const int F = a.F[r];
  if (threadIdx.x == 0) rs = merge_row(a, b, slot);
  if (threadIdx.x < 32) merge_topf(a, b, slot, F, S);
  __syncthreads();
  const RowStat R = rs;
  if (threadIdx.x == 0) {
    float sq = 0.f;
    if (!a.greedy)
      for (int i = 0; i < F; ++i)
        if (S[i]) sq = __fadd_rn(sq, ex2(__fmul_rn(__fsub_rn(cand_val(S[i]), R.m), a.kT)));
    s_sq = a.greedy ? 0.f : __fdiv_rn(sq, R.s);
  }
  __syncthreads();
  const char *row = row_ptr(a, 1, b, r, E::kSize);
  int d;
  float qd;
  if (a.greedy) {
    d = R.amax;
    qd = 1.f;
  } else {
    WSaguaro wf;
    wf.md = R.m;
    wf.kT = a.kT;
    wf.C = a.C;
    wf.hasS = F > 0;
    wf.keyF = F > 0 ? S[F - 1] : 0ull;
    float W;
    d = block_inv_cdf<E>(nullptr, row, a.V, o.u_draft[static_cast<size_t>(b) * a.K + r], wf, &W, inv);
    const float zd = E::ld(row, d);
    const bool ins = F > 0 && cand_key(zd, d) >= S[F - 1];
    const float q = __fdiv_rn(ex2(__fmul_rn(__fsub_rn(zd, R.m), a.kT)), R.s);
    qd = __fdiv_rn(ins ? __fmul_rn(q, a.C) : q, norm_N(a.C, s_sq));
  }
  if (threadIdx.x == 0) {
    o.d_out[static_cast<size_t>(b) * a.K + r] = d;
    if (o.qd_out) o.qd_out[static_cast<size_t>(b) * a.K + r] = qd;
  }
}

// Writes the guesses of sequence b from its merged top-F lists (S rows 0..K).
SSD_DEV void write_guesses(const VocabArgs &a, const FinishOut &o, int b, const uint64_t *S,
                           const RowStat *rs, int dslot0) {
  const int sumF = a.foff[a.K + 1];
  for (int k = 0; k <= a.K; ++k) {
    const int F = a.F[k];
    const RowStat R = rs[dslot0 + k];
    for (int i = threadIdx.x; i < F; i += blockDim.x) {
      const uint64_t key = S[k * a.Fcap + i];
      o.guess[static_cast<size_t>(b) * sumF + a.foff[k] + i] = cand_idx(key);
      if (o.guess_q) {
        float q;
        if (a.greedy) q = (i == 0) ? 1.f : 0.f;
        else q = __fdiv_rn(ex2(__fmul_rn(__fsub_rn(cand_val(key), R.m), a.kT)), R.s);
        o.guess_q[static_cast<size_t>(b) * sumF + a.foff[k] + i] = q;
      }
    }
  }
}

// Verification (+ optional prediction and lookup): one CTA per sequence.
template <class E>
__global__ void __launch_bounds__(kFinishThreads) k_verify_finish(const VocabArgs a, const FinishOut o) {
  extern __shared__ __align__(16) uint8_t dsm[];
  uint64_t *S = reinterpret_cast<uint64_t *>(dsm);  // [(K+1) * Fcap]
  __shared__ SeqShared sh;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int K = a.K;
  // merged statistics of every row this kernel reads
  for (int t = tid; t <= K; t += blockDim.x) {
    sh.rs[o.tslot0 + t] = merge_row(a, b, o.tslot0 + t);
    sh.rs[o.dslot0 + t] = merge_row(a, b, o.dslot0 + t);
  }
  for (int r = warp; r <= K; r += blockDim.x / 32) merge_topf(a, b, o.dslot0 + r, a.F[r], S + r * a.Fcap);
  __syncthreads();
  // per position j = t + 1: sum of q over S_j, p(d_j), q'(d_j), acceptance probability
  for (int t = tid; t <= K; t += blockDim.x) {
    const RowStat D = sh.rs[o.dslot0 + t];
    float sq = 0.f;
    if (!a.greedy)
      for (int i = 0; i < a.F[t]; ++i) {
        const uint64_t key = S[t * a.Fcap + i];
        if (key) sq = __fadd_rn(sq, ex2(__fmul_rn(__fsub_rn(cand_val(key), D.m), a.kT)));
      }
    sh.sq[t] = a.greedy ? 0.f : __fdiv_rn(sq, D.s);
  }
  __syncthreads();
  for (int t = tid; t < K; t += blockDim.x) {
    const int d = o.d_in[static_cast<size_t>(b) * K + t];
    const RowStat Tr = sh.rs[o.tslot0 + t], D = sh.rs[o.dslot0 + t];
    float p = 0.f, q = 0.f;
    if (d >= 0 && d < a.V) {
      const float zt = E::ld(row_ptr(a, 0, b, t, E::kSize), d);
      const float zd = E::ld(row_ptr(a, 1, b, t, E::kSize), d);
      if (a.greedy) {
        p = (d == Tr.amax) ? 1.f : 0.f;
        q = (d == D.amax) ? 1.f : 0.f;
      } else {
        const int F = a.F[t];
        const bool ins = F > 0 && cand_key(zd, d) >= S[t * a.Fcap + F - 1];
        p = __fdiv_rn(ex2(__fmul_rn(__fsub_rn(zt, Tr.m), a.kT)), Tr.s);
        const float qq = __fdiv_rn(ex2(__fmul_rn(__fsub_rn(zd, D.m), a.kT)), D.s);
        q = __fdiv_rn(ins ? __fmul_rn(qq, a.C) : qq, norm_N(a.C, sh.sq[t]));
      }
    } else {
      p = -1.f;  // marks an invalid token
      atomicOr(a.status, kFlagBadToken);
    }
    sh.p[t] = p;
    sh.qp[t] = q;
    if (o.accept_prob) {
      float ap;
      if (p < 0.f) ap = 0.f;
      else if (q > 0.f) ap = fminf(1.f, __fdiv_rn(p, q));
      else ap = (p > 0.f) ? 1.f : 0.f;
      o.accept_prob[static_cast<size_t>(b) * K + t] = ap;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int t = 0; t < K; ++t) {
      const float p = sh.p[t], q = sh.qp[t];
      const float u = o.u_acc[static_cast<size_t>(b) * K + t];
      if (p >= 0.f && __fmul_rn(u, q) < p) ++acc;
      else break;
    }
    sh.acc_len = acc;
  }
  __syncthreads();
  const int acc = sh.acc_len;
  // bonus token from row acc (position acc + 1)
  const RowStat Tr = sh.rs[o.tslot0 + acc];
  const char *rowT = row_ptr(a, 0, b, acc, E::kSize);
  const float ub = o.u_bonus[b];
  int bt;
  float W;
  bool zero_resid = false;
  if (acc < K) {
    const RowStat D = sh.rs[o.dslot0 + acc];
    if (a.greedy) {
      W = (Tr.amax != D.amax) ? 1.f : 0.f;
      zero_resid = !(W > 0.f);
      bt = Tr.amax;
    } else {
      const char *rowD = row_ptr(a, 1, b, acc, E::kSize);
      const int F = a.F[acc];
      WResidual wf;
      wf.mt = Tr.m;
      wf.kT = a.kT;
      wf.inv_st = __frcp_rn(Tr.s);
      wf.md = D.m;
      const float sN = __fmul_rn(D.s, norm_N(a.C, sh.sq[acc]));
      wf.f1 = __frcp_rn(sN);
      wf.fC = __fdiv_rn(a.C, sN);
      wf.hasS = F > 0;
      wf.keyF = F > 0 ? S[acc * a.Fcap + F - 1] : 0ull;
      bt = block_inv_cdf<E>(rowT, rowD, a.V, ub, wf, &W, sh.inv);
      if (bt < 0) {
        zero_resid = true;
        WTarget wp{Tr.m, a.kT};
        float Wp;
        bt = block_inv_cdf<E>(rowT, nullptr, a.V, ub, wp, &Wp, sh.inv);
      }
    }
  } else {
    W = 1.f;
    if (a.greedy) {
      bt = Tr.amax;
    } else {
      WTarget wp{Tr.m, a.kT};
      float Wp;
      bt = block_inv_cdf<E>(rowT, nullptr, a.V, ub, wp, &Wp, sh.inv);
    }
  }
  if (tid == 0) {
    if (zero_resid) atomicOr(a.status, kFlagZeroResidual);
    o.accept_len[b] = acc;
    o.bonus[b] = bt;
    for (int t = 0; t <= K; ++t) {
      int v = -1;
      if (t < acc) v = o.d_in[static_cast<size_t>(b) * K + t];
      if (t == acc) v = bt;
      o.out_tokens[static_cast<size_t>(b) * (K + 1) + t] = v;
    }
    if (o.resid_mass) o.resid_mass[b] = W;
  }
  // optional: guesses and cache lookup (the fused round)
  if (o.guess) {
    write_guesses(a, o, b, S, sh.rs, o.dslot0);
    if (tid == 0 && (o.slot || o.next_tokens || o.hits)) {
      const int F = a.F[acc];
      int s = -1;
      for (int i = 0; i < F; ++i)
        if (cand_idx(S[acc * a.Fcap + i]) == bt) {
          s = a.foff[acc] + i;
          break;
        }
      if (o.slot) o.slot[b] = s;
      if (o.next_tokens)
        for (int t = 0; t < K; ++t)
          o.next_tokens[static_cast<size_t>(b) * K + t] =
              (s >= 0 && o.payload) ? o.payload[(static_cast<size_t>(b) * a.foff[K + 1] + s) * K + t] : -1;
      if (o.hits && s >= 0) atomicAdd(o.hits, 1u);
    }
  }
}

// Outcome prediction alone: one CTA per sequence.
template <class E>
__global__ void __launch_bounds__(kFinishThreads) k_predict_finish(const VocabArgs a, const FinishOut o) {
  extern __shared__ __align__(16) uint8_t dsm[];
  uint64_t *S = reinterpret_cast<uint64_t *>(dsm);
  __shared__ RowStat rs[kMaxK + 1];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  for (int t = threadIdx.x; t <= a.K; t += blockDim.x) rs[t] = merge_row(a, b, o.dslot0 + t);
  for (int r = warp; r <= a.K; r += blockDim.x / 32) merge_topf(a, b, o.dslot0 + r, a.F[r], S + r * a.Fcap);
  __syncthreads();
  write_guesses(a, o, b, S, rs, 0);
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
  __shared__ float red[8];
  int h = 0;
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
  // integer counts are exact in float up to 2^24 sequences per call
  const float tot = block_sum<256>(static_cast<float>(h), red);
  if (threadIdx.x == 0 && l.hits) *l.hits = static_cast<uint32_t>(tot);
}

}  // namespace ssd

// ===========================================================================
// host side: validation, workspace layout, launches
// ===========================================================================
using namespace ssd;

namespace {

struct Layout {
  int nslots, nchunks, chunk_elems, Fcap;
  size_t stats_off, cands_off, total;
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
  const int tile = kFinishThreads * (dt == SSD_F32 ? EF32::kVec : EBF16::kVec);
  if ((V + tile - 1) / tile > kMaxTiles) return false;
  L->Fcap = fmax > 0 ? fmax : 1;
  const size_t nrec = static_cast<size_t>(B > 0 ? B : 1) * L->nslots * L->nchunks;
  L->stats_off = 0;
  L->cands_off = align_up(nrec * sizeof(ChunkStat), 256);
  L->total = align_up(L->cands_off + nrec * L->Fcap * sizeof(uint64_t), 256);
  return true;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssd_status_t check_logits(const void *p, ssd_dtype_t dt, int64_t seq_stride, int64_t row_stride, int B,
                          int K, int V) {
  if (B == 0) return SSD_OK;
  if (!p) return SSD_ERR_INVALID_ARG;
  if (row_stride < V && K > 0) return SSD_ERR_INVALID_ARG;
  if (seq_stride < 0 || row_stride < 0) return SSD_ERR_INVALID_ARG;
  if (B > 1 && seq_stride == 0) {
    // broadcasting one sequence to all is allowed (read-only)
  }
  const int es = esize(dt);
  if (!aligned16(p) || (seq_stride * es) % 16 || (row_stride * es) % 16) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

ssd_status_t check_common(ssd_dtype_t dt, int64_t seq_stride, int64_t row_stride, int B, int K, int V,
                          const int32_t *F, float C, float T, const Layout &L, void *ws, size_t ws_bytes,
                          bool needC) {
  (void)dt;
  (void)seq_stride;
  (void)row_stride;
  (void)B;
  (void)K;
  (void)V;
  (void)F;
  if (!(T >= 0.f) || !isfinite(T)) return SSD_ERR_INVALID_ARG;
  if (needC && !(C > 0.f && C <= 1.f)) return SSD_ERR_INVALID_ARG;
  if (B > 0 && (!ws || ws_bytes < L.total)) return SSD_ERR_WORKSPACE;
  if (B > 0 && !aligned16(ws)) return SSD_ERR_INVALID_ARG;
  return SSD_OK;
}

VocabArgs base_args(const void *target, const void *draft, int64_t seq_stride, int64_t row_stride, int B,
                    int K, int V, const int32_t *F, float C, float T, const Layout &L, void *ws,
                    uint32_t *status) {
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
  a.stats = reinterpret_cast<ChunkStat *>(static_cast<char *>(ws) + L.stats_off);
  a.cands = reinterpret_cast<uint64_t *>(static_cast<char *>(ws) + L.cands_off);
  a.status = status;
  return a;
}

// Optional timing hook (ssd_set_timing_events): events recorded around the
// statistics pass of every vocabulary call while set.
cudaEvent_t g_ev_before = nullptr;
cudaEvent_t g_ev_after = nullptr;

template <class E>
cudaError_t launch_stats_raw(const VocabArgs &a, cudaStream_t s);

template <class E>
cudaError_t launch_stats(const VocabArgs &a, cudaStream_t s) {
  if (g_ev_before) cudaEventRecord(g_ev_before, s);
  cudaError_t e = launch_stats_raw<E>(a, s);
  if (g_ev_after) cudaEventRecord(g_ev_after, s);
  return e;
}

template <class E>
cudaError_t launch_stats_raw(const VocabArgs &a, cudaStream_t s) {
  const size_t smem = kStages * kChunkBytes + kCandCap * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(k_row_stats<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long total = static_cast<long>(a.B) * a.nslots * a.nchunks;
  long grid = static_cast<long>(num_sms()) * 3;
  if (grid > total) grid = total;
  if (grid < 1) return cudaSuccess;
  k_row_stats<E><<<static_cast<unsigned>(grid), kStatsThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <class E>
cudaError_t launch_sample_finish(const VocabArgs &a, const FinishOut &o, cudaStream_t s) {
  if (a.K == 0 || a.B == 0) return cudaSuccess;
  const size_t smem = a.Fcap * sizeof(uint64_t);
  dim3 grid(a.K, a.B);
  k_sample_finish<E><<<grid, kFinishThreads, smem, s>>>(a, o);
  return cudaGetLastError();
}

template <class E>
cudaError_t launch_verify_finish(const VocabArgs &a, const FinishOut &o, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.K + 1) * a.Fcap * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(k_verify_finish<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k_verify_finish<E><<<a.B, kFinishThreads, smem, s>>>(a, o);
  return cudaGetLastError();
}

template <class E>
cudaError_t launch_predict_finish(const VocabArgs &a, const FinishOut &o, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.K + 1) * a.Fcap * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(k_predict_finish<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k_predict_finish<E><<<a.B, kFinishThreads, smem, s>>>(a, o);
  return cudaGetLastError();
}

ssd_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

void set_slots_verify(VocabArgs &a) {
  a.nslots = 2 * (a.K + 1);
  for (int r = 0; r <= a.K; ++r) {
    a.slot[r] = RowSlot{0, static_cast<int16_t>(r), 0, 0};
    a.slot[a.K + 1 + r] = RowSlot{1, static_cast<int16_t>(r), static_cast<int16_t>(a.F[r]), 0};
  }
}

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

size_t ssd_workspace_size(int B, int K, int V, ssd_dtype_t dt, const int32_t *F) {
  Layout L;
  if (!make_layout(B, K, V, dt, F, &L)) return 0;
  return L.total;
}

ssd_status_t ssd_saguaro_sample(const void *draft, ssd_dtype_t dt, int64_t seq_stride, int64_t row_stride,
                                int B, int K, int V, const int32_t *F, float C, float T,
                                const float *u_draft, int32_t *d_out, float *qd_out, uint32_t *status,
                                void *ws, size_t ws_bytes, ssd_stream_t s) {
  Layout L;
  if (!F || !make_layout(B, K, V, dt, F, &L)) return (F && B >= 0 && K >= 0 && V >= 1) ? SSD_ERR_UNSUPPORTED : SSD_ERR_INVALID_ARG;
  ssd_status_t st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(dt, seq_stride, row_stride, B, K, V, F, C, T, L, ws, ws_bytes, true);
  if (st != SSD_OK) return st;
  if (B == 0 || K == 0) return SSD_OK;
  if (!u_draft || !d_out || !status) return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(draft, draft, seq_stride, row_stride, B, K, V, F, C, T, L, ws, status);
  a.nslots = K;
  for (int r = 0; r < K; ++r) a.slot[r] = RowSlot{1, static_cast<int16_t>(r), static_cast<int16_t>(F[r]), 0};
  FinishOut o;
  memset(&o, 0, sizeof(o));
  o.u_draft = u_draft;
  o.d_out = d_out;
  o.qd_out = qd_out;
  o.dslot0 = 0;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  cudaError_t e;
  if (dt == SSD_F32) {
    e = launch_stats<EF32>(a, cs);
    if (e == cudaSuccess) e = launch_sample_finish<EF32>(a, o, cs);
  } else {
    e = launch_stats<EBF16>(a, cs);
    if (e == cudaSuccess) e = launch_sample_finish<EBF16>(a, o, cs);
  }
  return cuda_status(e);
}

ssd_status_t ssd_verify(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                        int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                        const int32_t *d, const float *u_acc, const float *u_bonus, int32_t *accept_len,
                        int32_t *out_tokens, int32_t *bonus, float *accept_prob, float *resid_mass,
                        uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s) {
  Layout L;
  if (!F || !make_layout(B, K, V, dt, F, &L)) return (F && B >= 0 && K >= 0 && V >= 1) ? SSD_ERR_UNSUPPORTED : SSD_ERR_INVALID_ARG;
  ssd_status_t st = check_logits(target, dt, seq_stride, row_stride, B, K, V);
  if (st == SSD_OK) st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(dt, seq_stride, row_stride, B, K, V, F, C, T, L, ws, ws_bytes, true);
  if (st != SSD_OK) return st;
  if (B == 0) return SSD_OK;
  if ((K > 0 && (!d || !u_acc)) || !u_bonus || !accept_len || !out_tokens || !bonus || !status)
    return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(target, draft, seq_stride, row_stride, B, K, V, F, C, T, L, ws, status);
  set_slots_verify(a);
  FinishOut o;
  memset(&o, 0, sizeof(o));
  o.d_in = d;
  o.u_acc = u_acc;
  o.u_bonus = u_bonus;
  o.accept_len = accept_len;
  o.out_tokens = out_tokens;
  o.bonus = bonus;
  o.accept_prob = accept_prob;
  o.resid_mass = resid_mass;
  o.tslot0 = 0;
  o.dslot0 = K + 1;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  cudaError_t e;
  if (dt == SSD_F32) {
    e = launch_stats<EF32>(a, cs);
    if (e == cudaSuccess) e = launch_verify_finish<EF32>(a, o, cs);
  } else {
    e = launch_stats<EBF16>(a, cs);
    if (e == cudaSuccess) e = launch_verify_finish<EBF16>(a, o, cs);
  }
  return cuda_status(e);
}

ssd_status_t ssd_predict_outcomes(const void *draft, ssd_dtype_t dt, int64_t seq_stride, int64_t row_stride,
                                  int B, int K, int V, const int32_t *F, float T, int32_t *guess,
                                  float *guess_q, uint32_t *status, void *ws, size_t ws_bytes,
                                  ssd_stream_t s) {
  Layout L;
  if (!F || !make_layout(B, K, V, dt, F, &L)) return (F && B >= 0 && K >= 0 && V >= 1) ? SSD_ERR_UNSUPPORTED : SSD_ERR_INVALID_ARG;
  ssd_status_t st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(dt, seq_stride, row_stride, B, K, V, F, 1.f, T, L, ws, ws_bytes, false);
  if (st != SSD_OK) return st;
  if (B == 0) return SSD_OK;
  if (!guess || !status) return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(draft, draft, seq_stride, row_stride, B, K, V, F, 1.f, T, L, ws, status);
  a.nslots = K + 1;
  for (int r = 0; r <= K; ++r) a.slot[r] = RowSlot{1, static_cast<int16_t>(r), static_cast<int16_t>(F[r]), 0};
  FinishOut o;
  memset(&o, 0, sizeof(o));
  o.guess = guess;
  o.guess_q = guess_q;
  o.dslot0 = 0;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  cudaError_t e;
  if (dt == SSD_F32) {
    e = launch_stats<EF32>(a, cs);
    if (e == cudaSuccess) e = launch_predict_finish<EF32>(a, o, cs);
  } else {
    e = launch_stats<EBF16>(a, cs);
    if (e == cudaSuccess) e = launch_predict_finish<EBF16>(a, o, cs);
  }
  return cuda_status(e);
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
                       int32_t *d_out, float *qd_out, int32_t *accept_len, int32_t *out_tokens,
                       int32_t *bonus, float *accept_prob, float *resid_mass, int32_t *guess,
                       float *guess_q, int32_t *slot, int32_t *next_tokens, uint32_t *hits,
                       uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s) {
  Layout L;
  if (!F || !make_layout(B, K, V, dt, F, &L)) return (F && B >= 0 && K >= 0 && V >= 1) ? SSD_ERR_UNSUPPORTED : SSD_ERR_INVALID_ARG;
  ssd_status_t st = check_logits(target, dt, seq_stride, row_stride, B, K, V);
  if (st == SSD_OK) st = check_logits(draft, dt, seq_stride, row_stride, B, K, V);
  if (st != SSD_OK) return st;
  st = check_common(dt, seq_stride, row_stride, B, K, V, F, C, T, L, ws, ws_bytes, true);
  if (st != SSD_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  if (hits) {
    cudaError_t e = cudaMemsetAsync(hits, 0, sizeof(uint32_t), cs);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
  }
  if (B == 0) return SSD_OK;
  if ((K > 0 && (!u_draft || !u_acc || !d_out)) || !u_bonus || !accept_len || !out_tokens || !bonus ||
      !status)
    return SSD_ERR_INVALID_ARG;
  if ((slot || next_tokens || hits) && !guess) return SSD_ERR_INVALID_ARG;
  VocabArgs a = base_args(target, draft, seq_stride, row_stride, B, K, V, F, C, T, L, ws, status);
  set_slots_verify(a);
  FinishOut o;
  memset(&o, 0, sizeof(o));
  o.u_draft = u_draft;
  o.d_out = d_out;
  o.qd_out = qd_out;
  o.d_in = d_out;
  o.u_acc = u_acc;
  o.u_bonus = u_bonus;
  o.accept_len = accept_len;
  o.out_tokens = out_tokens;
  o.bonus = bonus;
  o.accept_prob = accept_prob;
  o.resid_mass = resid_mass;
  o.guess = guess;
  o.guess_q = guess_q;
  o.payload = payload;
  o.slot = slot;
  o.next_tokens = next_tokens;
  o.hits = hits;
  o.tslot0 = 0;
  o.dslot0 = K + 1;
  cudaError_t e;
  if (dt == SSD_F32) {
    e = launch_stats<EF32>(a, cs);
    if (e == cudaSuccess) e = launch_sample_finish<EF32>(a, o, cs);
    if (e == cudaSuccess) e = launch_verify_finish<EF32>(a, o, cs);
  } else {
    e = launch_stats<EBF16>(a, cs);
    if (e == cudaSuccess) e = launch_sample_finish<EBF16>(a, o, cs);
    if (e == cudaSuccess) e = launch_verify_finish<EBF16>(a, o, cs);
  }
  return cuda_status(e);
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
