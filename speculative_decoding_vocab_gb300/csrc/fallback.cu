// fallback.cu -- the miss fallback of a speculation round on sm_103a.
//
// When the verification outcome of a sequence is not in the speculation
// cache, the round falls back to synchronous speculation with a backup
// speculator, and one miss holds up the whole batch for the backup's latency
// (technical summary "超越传统SD：SSD框架全异步解码实现4.7倍平均加速",
// "Saguaro 算法" part 3 "大 Batch 下的退避策略").  At large batch the pages
// switch to a backup of almost no latency: random tokens or an n-gram lookup.
// Two kernels serve that policy:
//
//   k_ngram_backup   one CTA per sequence; a missed sequence searches its own
//                    token history for the latest earlier occurrence of its
//                    last n tokens and proposes what followed, else uniform
//                    random tokens.  The scan runs backwards in chunks of
//                    4096 candidate positions (16 coalesced first-token loads
//                    in flight per thread), stops at the first chunk with a
//                    match, and checks the other n - 1 tokens only where the
//                    first one matches.
//   k_fallback_plan  one CTA of 128 threads; fp64 reduction over the batch of the hit
//                    probabilities and expected tokens into the expected round
//                    time, tokens, throughput and speedup of each backup, and
//                    the best backup -- on the device, so a chained backup
//                    call can act on it without a host round trip.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/ssd.h"
#include "common.cuh"

namespace {

using namespace ssd;

constexpr int kNgThreads = 256;
constexpr int kNgUnroll = 16;                        // first tokens in flight per thread
constexpr int kNgChunk = kNgThreads * kNgUnroll;     // candidate positions per pass
constexpr int kMaxN = 32;                            // longest n-gram
constexpr int kMaxBackupK = 1024;                    // longest proposal
constexpr int64_t kMaxHistory = int64_t(1) << 30;    // longest history row
constexpr int kPlanThreads = 128;  // fp64 is a slow pipe on this part: few threads, little reduction
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kMaxOptions = 8;

struct NgramArgs {
  const int32_t *hist;
  int64_t stride;
  const int32_t *hist_len;
  int n, K, V;
  const int32_t *slot;
  const float *u_rand;
  const int32_t *plan_best;
  int random_option;
  int32_t *next_tokens;
  int32_t *match_pos;
  uint32_t *status;
};

// floor(u V) for u in [0, 1), exactly: u * 2^24 is exact in fp32 and its
// integer part m gives (m V) >> 24.  u outside [0, 1) is clamped.
__device__ __forceinline__ int32_t random_token(float u, int V) {
  if (!(u >= 0.f)) u = 0.f;
  const unsigned long long m = static_cast<unsigned long long>(u * 16777216.0f);
  const unsigned long long t = (m * static_cast<unsigned long long>(V)) >> 24;
  return t >= static_cast<unsigned long long>(V) ? V - 1 : static_cast<int32_t>(t);
}

__global__ void __launch_bounds__(kNgThreads) k_ngram_backup(NgramArgs a) {
  __shared__ int32_t suf[kMaxN];
  __shared__ int red[2][kNgThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x;
  if (a.slot && a.slot[b] >= 0) {  // a hit keeps the cached tokens
    if (tid == 0 && a.match_pos) a.match_pos[b] = -2;
    return;
  }
  uint32_t fl = 0;
  const int n = a.n;
  const int32_t *h = a.hist ? a.hist + static_cast<int64_t>(b) * a.stride : nullptr;
  int L = a.hist_len ? a.hist_len[b] : 0;
  if (L < 0 || static_cast<int64_t>(L) > a.stride) {
    if (n >= 1) fl |= kFlagBadHistory;
    L = 0;
  }
  bool search = n >= 1 && L >= n + 1;
  if (search && a.plan_best && *a.plan_best == a.random_option) search = false;

  int m = -1;
  if (search) {
    if (tid < n) suf[tid] = h[L - n + tid];
    __syncthreads();
    const int32_t s0 = suf[0];
    // candidates c in [0, L - n): h[c .. c+n) == suffix, the largest wins
    int par = 0;
    for (int top = L - n; top > 0; top -= kNgChunk, par ^= 1) {
      int32_t first[kNgUnroll];
#pragma unroll
      for (int j = 0; j < kNgUnroll; ++j) {
        const int c = top - 1 - tid - kNgThreads * j;
        first[j] = c >= 0 ? __ldg(h + c) : ~s0;
      }
      int best = -1;
#pragma unroll
      for (int j = 0; j < kNgUnroll; ++j) {
        const int c = top - 1 - tid - kNgThreads * j;
        if (best < 0 && c >= 0 && first[j] == s0) {
          bool eq = true;
          for (int i = 1; i < n && eq; ++i) eq = __ldg(h + c + i) == suf[i];
          if (eq) best = c;
        }
      }
      best = __reduce_max_sync(0xffffffffu, best);
      if ((tid & 31) == 0) red[par][tid >> 5] = best;
      __syncthreads();
#pragma unroll
      for (int w = 0; w < kNgThreads / 32; ++w) m = max(m, red[par][w]);
      if (m >= 0) break;  // the same m in every thread: a uniform exit
    }
  }
  if (tid == 0 && a.match_pos) a.match_pos[b] = m;
  for (int t = tid; t < a.K; t += kNgThreads) {
    const int p = m + n + t;
    int32_t tok;
    if (m >= 0 && p < L) {
      tok = __ldg(h + p);
      if (tok < 0 || tok >= a.V) {
        fl |= kFlagBadToken;
        tok = random_token(a.u_rand[static_cast<int64_t>(b) * a.K + t], a.V);
      }
    } else {
      tok = random_token(a.u_rand[static_cast<int64_t>(b) * a.K + t], a.V);
    }
    a.next_tokens[static_cast<int64_t>(b) * a.K + t] = tok;
  }
  if (fl) atomicOr(a.status, fl);
}

struct PlanArgs {
  const float *p_hit, *e_hit;
  int B;
  double T_v, T_p;
  int nopt;
  double T_b[kMaxOptions], e_miss[kMaxOptions];
  double *time, *tokens, *throughput, *speedup;
  int32_t *best;
  uint32_t *status;
};

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_prod_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v *= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kPlanThreads) k_fallback_plan(PlanArgs a) {
  __shared__ double red[4][kPlanWarps];
  const int tid = threadIdx.x;
  double pall = 1.0, phe = 0.0, pmiss = 0.0, ehit = 0.0;
  uint32_t fl = 0;
  for (int b = tid; b < a.B; b += kPlanThreads) {
    double p = a.p_hit[b], e = a.e_hit[b];
    if (!(p >= 0.0 && p <= 1.0)) {
      fl |= kFlagBadRate;
      p = p > 1.0 ? 1.0 : 0.0;
    }
    if (!(e >= 0.0 && e <= 1e30)) {
      fl |= kFlagBadRate;
      e = 0.0;
    }
    pall *= p;
    phe += p * e;
    pmiss += 1.0 - p;
    ehit += e;
  }
  pall = warp_prod_d(pall);
  phe = warp_sum_d(phe);
  pmiss = warp_sum_d(pmiss);
  ehit = warp_sum_d(ehit);
  if ((tid & 31) == 0) {
    red[0][tid >> 5] = pall;
    red[1][tid >> 5] = phe;
    red[2][tid >> 5] = pmiss;
    red[3][tid >> 5] = ehit;
  }
  if (fl) atomicOr(a.status, fl);
  __syncthreads();
  if (tid < 32) {
    // one warp part per lane; the lanes past the warp count add the identities
    const bool has = tid < kPlanWarps;
    const int w = has ? tid : 0;  // every load in bounds
    pall = warp_prod_d(has ? red[0][w] : 1.0);
    phe = warp_sum_d(has ? red[1][w] : 0.0);
    pmiss = warp_sum_d(has ? red[2][w] : 0.0);
    ehit = warp_sum_d(has ? red[3][w] : 0.0);
    // one option per lane; the best is the largest throughput, lowest index on ties
    const double tmax = a.T_v > a.T_p ? a.T_v : a.T_p;
    const double base = ehit / (a.T_p + a.T_v);
    double thr = -1.0;
    if (tid < a.nopt) {
      const double time = tmax + (1.0 - pall) * a.T_b[tid];
      const double tokens = phe + pmiss * a.e_miss[tid];
      thr = tokens / time;
      if (a.time) a.time[tid] = time;
      if (a.tokens) a.tokens[tid] = tokens;
      if (a.throughput) a.throughput[tid] = thr;
      if (a.speedup) a.speedup[tid] = thr / base;
    }
    double mx = thr;
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const unsigned top = __ballot_sync(0xffffffffu, tid < a.nopt && thr == mx);
    if (tid == 0 && a.best) a.best[0] = __ffs(top) - 1;
  }
}

ssd_status_t cuda_rc(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

}  // namespace

extern "C" ssd_status_t ssd_ngram_backup(const int32_t *hist, int64_t hist_stride,
                                         const int32_t *hist_len, int B, int n, int K, int V,
                                         const int32_t *slot, const float *u_rand,
                                         const int32_t *plan_best, int random_option,
                                         int32_t *next_tokens, int32_t *match_pos,
                                         uint32_t *status, ssd_stream_t s) {
  if (B < 0 || n < 0 || K < 0 || V < 1) return SSD_ERR_INVALID_ARG;
  if (n > kMaxN || K > kMaxBackupK) return SSD_ERR_UNSUPPORTED;
  if (B == 0) return SSD_OK;
  if (!status || (K > 0 && (!next_tokens || !u_rand))) return SSD_ERR_INVALID_ARG;
  if (n >= 1 && (!hist || !hist_len || hist_stride < 1)) return SSD_ERR_INVALID_ARG;
  if (hist_stride > kMaxHistory) return SSD_ERR_UNSUPPORTED;  // positions stay int32
  NgramArgs a{hist, hist_stride, hist_len, n, K, V, slot, u_rand, plan_best, random_option,
              next_tokens, match_pos, status};
  k_ngram_backup<<<B, kNgThreads, 0, reinterpret_cast<cudaStream_t>(s)>>>(a);
  return cuda_rc(cudaGetLastError());
}

extern "C" ssd_status_t ssd_fallback_plan(const float *p_hit, const float *e_hit, int B, double T_v,
                                          double T_p, int nopt, const double *T_b,
                                          const double *e_miss, double *time, double *tokens,
                                          double *throughput, double *speedup, int32_t *best,
                                          uint32_t *status, ssd_stream_t s) {
  if (B < 1 || nopt < 1 || !p_hit || !e_hit || !T_b || !e_miss || !status) return SSD_ERR_INVALID_ARG;
  if (nopt > kMaxOptions) return SSD_ERR_UNSUPPORTED;
  if (!(T_v >= 0.0) || !(T_p >= 0.0) || !(T_v + T_p > 0.0) || !isfinite(T_v + T_p))
    return SSD_ERR_INVALID_ARG;
  PlanArgs a{};
  a.p_hit = p_hit;
  a.e_hit = e_hit;
  a.B = B;
  a.T_v = T_v;
  a.T_p = T_p;
  a.nopt = nopt;
  for (int o = 0; o < nopt; ++o) {
    if (!(T_b[o] >= 0.0) || !isfinite(T_b[o]) || !(e_miss[o] >= 0.0) || !isfinite(e_miss[o]))
      return SSD_ERR_INVALID_ARG;
    a.T_b[o] = T_b[o];
    a.e_miss[o] = e_miss[o];
  }
  a.time = time;
  a.tokens = tokens;
  a.throughput = throughput;
  a.speedup = speedup;
  a.best = best;
  a.status = status;
  k_fallback_plan<<<1, kPlanThreads, 0, reinterpret_cast<cudaStream_t>(s)>>>(a);
  return cuda_rc(cudaGetLastError());
}
