// common.cuh -- device helpers shared by the sm_103a kernels of the
// speculation-round library: status bits, order-preserving keys, TMA bulk
// copies with mbarriers (bounded waits), and deterministic reductions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define SSD_DEV __device__ __forceinline__

namespace ssd {

// status-word bits (mirror include/ssd.h)
constexpr uint32_t kFlagBadToken = 1u;
constexpr uint32_t kFlagZeroResidual = 2u;
constexpr uint32_t kFlagWaitTimeout = 4u;
constexpr uint32_t kFlagBadOutcome = 8u;
constexpr uint32_t kFlagBadTree = 16u;
constexpr uint32_t kFlagBadBlock = 32u;
constexpr uint32_t kFlagBadPrefix = 64u;
constexpr uint32_t kFlagBadHistory = 128u;
constexpr uint32_t kFlagBadRate = 256u;

// Upper bound on polls of an mbarrier before a wait gives up and reports
// SSD_FLAG_WAIT_TIMEOUT (each poll may suspend the thread for a short,
// hardware-defined time; copies here finish in microseconds).
constexpr uint32_t kMaxPolls = 1u << 22;

SSD_DEV uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Asynchronous global -> shared copies (all in flight together; one wait).
// 16 bytes through L2 only; 8 and 4 bytes through L1 (callers order them
// after the acquire that makes the source current).
SSD_DEV void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
SSD_DEV void cp_async8(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
SSD_DEV void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
SSD_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---------------------------------------------------------------------------
// order-preserving keys: larger float -> larger unsigned key
// ---------------------------------------------------------------------------
SSD_DEV uint32_t f2ord(float f) {
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
SSD_DEV float ord2f(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}
// Candidate key ranking (value descending, index ascending) as one unsigned
// 64-bit number: the larger key is the better candidate.  Key 0 is the
// "no candidate" sentinel (it decodes to index -1).
SSD_DEV uint64_t cand_key(float v, int idx) {
  return (static_cast<uint64_t>(f2ord(v)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}
SSD_DEV float cand_val(uint64_t k) { return ord2f(static_cast<uint32_t>(k >> 32)); }
SSD_DEV int cand_idx(uint64_t k) { return static_cast<int>(~static_cast<uint32_t>(k)); }

// 2^x on the SFU (ex2.approx, flush-to-zero); deterministic for equal inputs.
SSD_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// mbarrier + TMA bulk copy (global -> shared)
// ---------------------------------------------------------------------------
SSD_DEV void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
SSD_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
SSD_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
SSD_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
SSD_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// One poll that may suspend the thread for up to `ns` nanoseconds while the
// phase is incomplete (no busy spinning).
SSD_DEV bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity; false on timeout.
SSD_DEV bool mbar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t it = 0; it < kMaxPolls; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// The same wait for a single thread that may sleep between polls (at most
// kMaxPolls polls of at most 1 us each).
SSD_DEV bool mbar_wait_sleep(uint64_t *bar, uint32_t parity) {
  for (uint32_t it = 0; it < kMaxPolls; ++it)
    if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
  return false;
}
// One bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
// completing on `bar`'s transaction count.
SSD_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// packed arithmetic: two fp32 lanes in a 64-bit register (Blackwell FMA2 /
// ADD2), two bf16 lanes in a 32-bit register
// ---------------------------------------------------------------------------
SSD_DEV uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
SSD_DEV void unpack2(uint64_t v, float &lo, float &hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
SSD_DEV uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {  // a * b + c per lane, round to nearest
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
SSD_DEV uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
SSD_DEV uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
SSD_DEV uint32_t bmax2(uint32_t a, uint32_t b) {  // lane-wise maximum of two bf16 pairs
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---------------------------------------------------------------------------
// element types of the logits
// ---------------------------------------------------------------------------
struct EF32 {
  static constexpr int kVec = 4;  // elements per 16-byte vector
  static constexpr int kSize = 4;
  static constexpr int kLowBit = 0;  // lowest key bit that can differ
  SSD_DEV static void unpack(const uint4 &w, float *f) {
    f[0] = __uint_as_float(w.x);
    f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z);
    f[3] = __uint_as_float(w.w);
  }
  SSD_DEV static float ld(const void *base, int64_t i) {
    return __ldg(reinterpret_cast<const float *>(base) + i);
  }
  static constexpr int kPairs = 2;  // packed fp32 pairs per vector
  SSD_DEV static uint64_t pair(const uint4 &w, int h) {
    return h == 0 ? pack2(__uint_as_float(w.x), __uint_as_float(w.y)) : pack2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
};
struct EBF16 {
  static constexpr int kVec = 8;
  static constexpr int kSize = 2;
  static constexpr int kLowBit = 16;  // a bf16 value's float key has constant low 16 bits
  SSD_DEV static void unpack(const uint4 &w, float *f) {
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xFFFF0000u);
    f[4] = __uint_as_float(w.z << 16);
    f[5] = __uint_as_float(w.z & 0xFFFF0000u);
    f[6] = __uint_as_float(w.w << 16);
    f[7] = __uint_as_float(w.w & 0xFFFF0000u);
  }
  SSD_DEV static float ld(const void *base, int64_t i) {
    uint16_t h = __ldg(reinterpret_cast<const unsigned short *>(base) + i);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  static constexpr int kPairs = 4;
  SSD_DEV static uint64_t pair(const uint4 &w, int h) {
    const uint32_t x = h == 0 ? w.x : (h == 1 ? w.y : (h == 2 ? w.z : w.w));
    return pack2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
  }
};

// Load VEC consecutive elements starting at i0 of a row of length V; lanes
// past the end read as -inf and are flagged invalid.
template <class E>
SSD_DEV void load_vec(const void *row, int i0, int V, float *f, bool *valid) {
  if (i0 + E::kVec <= V) {
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(
        reinterpret_cast<const char *>(row) + static_cast<int64_t>(i0) * E::kSize));
    E::unpack(w, f);
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) valid[e] = true;
  } else {
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) {
      valid[e] = (i0 + e) < V;
      f[e] = valid[e] ? E::ld(row, i0 + e) : -__int_as_float(0x7f800000);
    }
  }
}

// ---------------------------------------------------------------------------
// barrier of a group of NT threads (named barrier 1): the first NT threads of a
// CTA synchronise without the CTA's other warps
// ---------------------------------------------------------------------------
template <int NT>
SSD_DEV void group_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
template <int NT>
SSD_DEV int group_sync_count(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "bar.red.popc.u32 %0, 1, %2, p;\n\t}\n"
      : "=r"(r)
      : "r"(pred), "n"(NT)
      : "memory");
  return r;
}
template <int NT>
SSD_DEV int group_sync_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred), "n"(NT)
      : "memory");
  return r;
}

// ---------------------------------------------------------------------------
// deterministic warp / block reductions (fixed association order); "block"
// here is the group of the first NT threads (named barrier 1)
// ---------------------------------------------------------------------------
SSD_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
SSD_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
SSD_DEV uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = (w > v) ? w : v;
  }
  return v;
}

// Every thread receives the block maximum.  `red` holds >= NT/32 floats.
template <int NT>
SSD_DEV float block_max(float v, float *red) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  group_sync<NT>();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = fmaxf(r, red[w]);
  group_sync<NT>();
  return r;
}
// Every thread receives the same block sum (lane 0 of each warp, warps in order).
template <int NT>
SSD_DEV float block_sum(float v, float *red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  group_sync<NT>();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = __fadd_rn(r, red[w]);
  group_sync<NT>();
  return r;
}
template <int NT>
SSD_DEV uint64_t block_max_u64(uint64_t v, uint64_t *red) {
  v = warp_max_u64(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  group_sync<NT>();
  uint64_t r = red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = (red[w] > r) ? red[w] : r;
  group_sync<NT>();
  return r;
}

// Exclusive prefix sum of one float per thread, in thread order, with a fixed
// association: warp-level Hillis-Steele scan, then the warp totals scanned by
// one thread.  Returns the exclusive prefix; `red` holds >= NT/32 + 1 floats.
template <int NT>
SSD_DEV float block_excl_scan(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc = __fadd_rn(inc, t);
  }
  float excl_lane = __shfl_up_sync(0xffffffffu, inc, 1);
  if (lane == 0) excl_lane = 0.f;
  if (lane == 31) red[warp] = inc;
  group_sync<NT>();
  if (threadIdx.x == 0) {
    float run = 0.f;
    for (int w = 0; w < NT / 32; ++w) {
      float t = red[w];
      red[w] = run;
      run = __fadd_rn(run, t);
    }
    red[NT / 32] = run;
  }
  group_sync<NT>();
  float r = __fadd_rn(red[warp], excl_lane);
  group_sync<NT>();
  return r;
}

}  // namespace ssd
