// fill.cu -- the tree K/V append of a branch-decode step on sm_103a.
//
// While the target verifies, the draft pre-speculates a continuation for
// every predicted outcome: it decodes all F_k branches together, one token
// per branch and step, over a tree-masked paged K/V cache (technical summary
// "超越传统SD：SSD框架全异步解码实现4.7倍平均加速", "投机解码的瓶颈与 SSD 的核心机制"
// and "工程优化与系统表现").  Each step appends the key and value rows of the
// tokens it feeds to the cache at their tree nodes' positions; the draw of
// the next token per branch is ssd_fill_sample (the vocabulary kernels).
//
//   k_kv_append  one thread per 16-byte vector of a (sequence, node, KV head)
//                row: coalesced reads of the new rows, writes of whole
//                16-byte pieces into the page the block table names.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssd.h"
#include "common.cuh"

namespace {

using namespace ssd;

constexpr int kAppendThreads = 256;
constexpr int kPage = 16;

struct AppendArgs {
  const uint4 *k_new, *v_new;
  uint4 *k_cache, *v_cache;
  const int32_t *block_table;
  int maxb;
  int64_t num_blocks;
  const int32_t *prefix_len;
  int node0, S, Hkv, vpr;  // vpr: 16-byte vectors per row (d / 8)
  int64_t total;           // B * S * Hkv * vpr
  uint32_t *status;
};

__global__ void __launch_bounds__(kAppendThreads) k_kv_append(AppendArgs a) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kAppendThreads + threadIdx.x;
  if (g >= a.total) return;
  const int e = static_cast<int>(g % a.vpr);
  const int64_t row = g / a.vpr;  // (b, i, h), h fastest
  const int h = static_cast<int>(row % a.Hkv);
  const int64_t bi = row / a.Hkv;
  const int i = static_cast<int>(bi % a.S);
  const int b = static_cast<int>(bi / a.S);
  const int pl = a.prefix_len[b];
  const int64_t pos = static_cast<int64_t>(pl) + a.node0 + i;
  if (pl < 0 || pos / kPage >= a.maxb) {
    if (e == 0) atomicOr(a.status, kFlagBadPrefix);
    return;
  }
  const int64_t blk = a.block_table[static_cast<int64_t>(b) * a.maxb + pos / kPage];
  if (blk < 0 || blk >= a.num_blocks) {
    if (e == 0) atomicOr(a.status, kFlagBadBlock);
    return;
  }
  const int64_t dst = ((blk * a.Hkv + h) * kPage + pos % kPage) * a.vpr + e;
  a.k_cache[dst] = a.k_new[g];
  a.v_cache[dst] = a.v_new[g];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" ssd_status_t ssd_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                      const int32_t *block_table, int maxb, int64_t num_blocks,
                                      const int32_t *prefix_len, int node0, int B, int S, int Hkv, int d,
                                      uint32_t *status, ssd_stream_t s) {
  if (B < 0 || S < 0 || Hkv < 1 || d < 1 || node0 < 0 || maxb < 1 || num_blocks < 1)
    return SSD_ERR_INVALID_ARG;
  if (d % 8 || d > 256) return SSD_ERR_UNSUPPORTED;
  if (B == 0 || S == 0) return SSD_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !prefix_len || !status)
    return SSD_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return SSD_ERR_UNSUPPORTED;
  AppendArgs a{};
  a.k_new = static_cast<const uint4 *>(k_new);
  a.v_new = static_cast<const uint4 *>(v_new);
  a.k_cache = static_cast<uint4 *>(k_cache);
  a.v_cache = static_cast<uint4 *>(v_cache);
  a.block_table = block_table;
  a.maxb = maxb;
  a.num_blocks = num_blocks;
  a.prefix_len = prefix_len;
  a.node0 = node0;
  a.S = S;
  a.Hkv = Hkv;
  a.vpr = d / 8;
  a.total = static_cast<int64_t>(B) * S * Hkv * a.vpr;
  a.status = status;
  const int64_t grid = (a.total + kAppendThreads - 1) / kAppendThreads;
  if (grid > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
  k_kv_append<<<static_cast<unsigned>(grid), kAppendThreads, 0, reinterpret_cast<cudaStream_t>(s)>>>(a);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
