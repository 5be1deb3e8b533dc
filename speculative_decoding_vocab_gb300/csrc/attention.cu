// attention.cu -- tree-masked decode attention over a paged bf16 KV cache
// (sm_103a), so the draft decodes every branch of the speculation tree in one
// forward pass: the "custom sparse attention mask" of the technical summary
// "超越传统SD：SSD框架全异步解码实现4.7倍平均加速", section "工程优化与系统表现".
//
// Row i of head h (query node m = N - Nq + i) sees every prefix position and
// the tree nodes on m's ancestor-or-self path; node n's K/V sits at logical
// position prefix_len + n.  GQA: head h reads KV head h / (Hq / Hkv).
//
// This file holds the CUDA-core kernel: one CTA per (sequence, KV head, block
// of 64 query rows) walks the sequence's KV pages, staging each 16-position
// page of K and V in shared memory, with an online (running-max) softmax in
// the log2 domain and fp32 accumulation.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "../../include/ssd.h"
#include "common.cuh"

namespace ssd {

constexpr int kPage = 16;
constexpr int kMaxNodes = 128;
constexpr int kAttnThreads = 256;
// query rows per CTA (8 warps): 64 at d = 64, 32 at d = 128 (static shared memory < 48 KiB)
template <int D>
struct RowsPerCta {
  static constexpr int value = D == 64 ? 64 : 32;
};

struct AttnArgs {
  const uint16_t *q, *k, *v;
  const int32_t *table;
  int maxb;
  int64_t num_blocks;
  const int32_t *prefix_len, *parent;
  int B, N, Nq, Hq, Hkv, d;
  float scale_log2;  // scale * log2(e)
  uint16_t *out;
  float *lse;
  uint32_t *status;
};

SSD_DEV float bf2f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }
SSD_DEV uint16_t f2bf(float f) {
  // round to nearest even (finite inputs)
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) k_branch_attn_simt(const AttnArgs a) {
  constexpr int kRowsPerCta = RowsPerCta<D>::value;
  constexpr int kRowsPerWarp = kRowsPerCta / (kAttnThreads / 32);
  __shared__ uint32_t anc[kMaxNodes][kMaxNodes / 32];  // ancestor-or-self bits per node
  __shared__ __align__(16) float qs[kRowsPerCta][D];
  __shared__ __align__(16) float ks[kPage][D + 1];
  __shared__ __align__(16) float vs[kPage][D];
  __shared__ int page_ok;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.Hkv, hk = blockIdx.x % a.Hkv;
  const int group = a.Hq / a.Hkv;
  const int nrows = group * a.Nq;
  const int row0 = blockIdx.y * kRowsPerCta;
  const int N = a.N;
  const int L = max(0, a.prefix_len[b]);
  const int nkeys = L + N;

  // ancestor masks
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
  // query rows of this CTA: row = node_local * group + g  (all heads of the group)
  for (int i = tid; i < kRowsPerCta * D; i += kAttnThreads) {
    const int r = i / D, e = i % D;
    const int row = row0 + r;
    float x = 0.f;
    if (row < nrows) {
      const int qi = row / group, h = hk * group + row % group;
      x = bf2f(a.q[((static_cast<int64_t>(b) * a.Nq + qi) * a.Hq + h) * D + e]);
    }
    qs[r][e] = x;
  }
  __syncthreads();

  constexpr int DPL = D / 32;  // output elements per lane
  float o[kRowsPerWarp][DPL];
  float mrun[kRowsPerWarp], lrun[kRowsPerWarp];
  const float NEG_INF = -__int_as_float(0x7f800000);
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    mrun[r] = NEG_INF;
    lrun[r] = 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) o[r][t] = 0.f;
  }

  const int npages = (nkeys + kPage - 1) / kPage;
  for (int p = 0; p < npages; ++p) {
    if (tid == 0) {
      const int blk = p < a.maxb ? a.table[static_cast<int64_t>(b) * a.maxb + p] : -1;
      page_ok = (blk >= 0 && blk < a.num_blocks) ? 1 : 0;
      if (!page_ok) atomicOr(a.status, kFlagBadBlock);
    }
    __syncthreads();
    const bool ok = page_ok != 0;
    if (ok) {
      const int blk = a.table[static_cast<int64_t>(b) * a.maxb + p];
      const uint16_t *kp = a.k + (static_cast<int64_t>(blk) * a.Hkv + hk) * kPage * D;
      const uint16_t *vp = a.v + (static_cast<int64_t>(blk) * a.Hkv + hk) * kPage * D;
      for (int i = tid; i < kPage * D; i += kAttnThreads) {
        ks[i / D][i % D] = bf2f(kp[i]);
        vs[i / D][i % D] = bf2f(vp[i]);
      }
    }
    __syncthreads();
    if (ok) {
      // lane handles key j = lane & 15 for rows in half (lane >> 4)
      const int j = lane & 15;
      const int pos = p * kPage + j;
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const int rl = warp * kRowsPerWarp + r;  // local row
        const int row = row0 + rl;
        // every lane computes the score of (row, key j) for its half of d; combine halves
        float acc = 0.f;
        const int e0 = (lane >> 4) * (D / 2);
#pragma unroll 8
        for (int e = 0; e < D / 2; ++e) acc = fmaf(qs[rl][e0 + e], ks[j][e0 + e], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 16);
        bool vis = row < nrows && pos < nkeys;
        if (vis && pos >= L) {
          const int node = N - a.Nq + row / group;
          const int n = pos - L;
          vis = (anc[node][n >> 5] >> (n & 31)) & 1u;
        }
        const float sc = vis ? acc * a.scale_log2 : NEG_INF;
        // running max over the 16 keys of the page
        float pm = sc;
#pragma unroll
        for (int off = 8; off; off >>= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, off));
        const float mnew = fmaxf(mrun[r], pm);
        if (mnew == NEG_INF) continue;  // nothing visible yet for this row
        const float alpha = ex2(mrun[r] - mnew);
        const float pj = vis ? ex2(sc - mnew) : 0.f;
        float ps = pj;
#pragma unroll
        for (int off = 8; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        lrun[r] = lrun[r] * alpha + ps;
        mrun[r] = mnew;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
          const int e = lane + 32 * t;
          float acc2 = o[r][t] * alpha;
#pragma unroll
          for (int jj = 0; jj < kPage; ++jj) {
            const float pjj = __shfl_sync(0xffffffffu, pj, jj);
            acc2 = fmaf(pjj, vs[jj][e], acc2);
          }
          o[r][t] = acc2;
        }
      }
    }
    __syncthreads();
  }
  // write out
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int rl = warp * kRowsPerWarp + r;
    const int row = row0 + rl;
    if (row >= nrows) continue;
    const int qi = row / group, h = hk * group + row % group;
    const float inv = lrun[r] > 0.f ? 1.f / lrun[r] : 0.f;
    uint16_t *op = a.out + ((static_cast<int64_t>(b) * a.Nq + qi) * a.Hq + h) * D;
#pragma unroll
    for (int t = 0; t < DPL; ++t) op[lane + 32 * t] = f2bf(o[r][t] * inv);
    if (a.lse && lane == 0)
      a.lse[(static_cast<int64_t>(b) * a.Nq + qi) * a.Hq + h] =
          lrun[r] > 0.f ? (mrun[r] + log2f(lrun[r])) * 0.69314718055994531f : NEG_INF;
  }
}

}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_attention_workspace_size(int B, int Nq, int Hq, int Hkv, int d, int max_prefix) {
  (void)B;
  (void)Nq;
  (void)Hq;
  (void)Hkv;
  (void)d;
  (void)max_prefix;
  return 0;
}

ssd_status_t ssd_branch_attention(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_table, int maxb, int64_t num_blocks,
                                  const int32_t *prefix_len, const int32_t *parent, int B, int N, int Nq,
                                  int Hq, int Hkv, int d, float scale, void *out, float *lse,
                                  uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s) {
  (void)ws;
  (void)ws_bytes;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || !(scale > 0.f) || !isfinite(scale)) return SSD_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return SSD_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SSD_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16 || N < 1 || N > kMaxNodes || Nq < 1 || Nq > N) return SSD_ERR_UNSUPPORTED;
  if (B == 0) return SSD_OK;
  if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !parent || !out || !status || maxb < 1 ||
      num_blocks < 1)
    return SSD_ERR_INVALID_ARG;
  AttnArgs a;
  a.q = static_cast<const uint16_t *>(q);
  a.k = static_cast<const uint16_t *>(k_cache);
  a.v = static_cast<const uint16_t *>(v_cache);
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
  a.d = d;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = static_cast<uint16_t *>(out);
  a.lse = lse;
  a.status = status;
  const int nrows = (Hq / Hkv) * Nq;
  const int rpc = d == 64 ? RowsPerCta<64>::value : RowsPerCta<128>::value;
  dim3 grid(B * Hkv, (nrows + rpc - 1) / rpc);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  if (d == 64) k_branch_attn_simt<64><<<grid, kAttnThreads, 0, cs>>>(a);
  else k_branch_attn_simt<128><<<grid, kAttnThreads, 0, cs>>>(a);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
