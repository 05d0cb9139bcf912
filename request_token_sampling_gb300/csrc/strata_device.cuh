// strata_device.cuh -- device-side building blocks of the GB300 sampler kernel.
//
// Inline PTX for the sm_103a features the kernel is built on: bulk (TMA) global->shared copies
// completed on an mbarrier, thread-block-cluster barriers and distributed shared memory (DSMEM)
// stores, programmatic dependent launch, and the warp-wide redux.  Plus the order key used by
// every selection, the penalty, and Philox4x32-10.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

// Branch hints for the rarely taken fallbacks of the post-pass: the compiler lays the common path
// out in one run, so a block fetches its instructions with fewer jumps.
#define STRATA_LIKELY(x) __builtin_expect(!!(x), 1)
#define STRATA_UNLIKELY(x) __builtin_expect(!!(x), 0)

namespace strata {

constexpr uint32_t FULL_MASK = 0xFFFFFFFFu;

// ------------------------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make this CTA's generic-proxy writes to shared memory (an mbarrier initialisation) visible to
// the async proxy (the bulk copies that complete on it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Make the mbarrier initialisation visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from global memory into
// this CTA's shared memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Arrive without release semantics: only marks this CTA as running (nothing to publish yet).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// Atomic add on a cluster CTA's shared memory word; returns the previous value.
__device__ __forceinline__ uint32_t dsmem_atomic_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void dsmem_st_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Asynchronous 16- / 8-byte store into a cluster CTA's shared memory; the bytes complete on that
// CTA's mbarrier `bar` (a shared::cluster address) as transaction bytes.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_async_v2(uint32_t addr, uint32_t a, uint32_t b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "r"(a), "r"(b), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t a, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr), "r"(a),
               "r"(bar)
               : "memory");
}

// One arrival on a cluster CTA's mbarrier that also announces `bytes` more transaction bytes.
// The bytes may land before or after the arrival: the phase completes once every expected
// arrival has happened and the transaction count is back to zero.
__device__ __forceinline__ void mbar_arrive_expect_tx_remote(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Plain local arrival (release at CTA scope: this thread's earlier shared-memory writes are seen
// by the threads that wait on the phase).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------------------------------------ PDL
// Hint: bring the line holding `p` (global memory) into L1.
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ------------------------------------------------------------------------------ arithmetic
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order key of a logit: unsigned order equals float order, -0 equals +0, NaN maps to 0 (below
// the key of -inf, 0x007FFFFF), so NaN ranks last and 0 can mean "no element".
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t b = __float_as_uint(v);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// 64-bit selection key: value order in the high word, lower index wins ties (complemented id).
__device__ __forceinline__ uint64_t sel_key(uint32_t ord, uint32_t id) {
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(~id);
}
__device__ __forceinline__ uint32_t key_id(uint64_t k) { return ~static_cast<uint32_t>(k); }

// The repeat / frequency / presence penalty of an id seen `count` > 0 times, IEEE float32 with
// one rounding per operation: repeat multiplies a non-positive logit and divides a positive one,
// then count*freq + present is subtracted.
__device__ __forceinline__ float penalize(float x, uint32_t count, float rep, float freq, float pres) {
  x = (x <= 0.0f) ? __fmul_rn(x, rep) : __fdiv_rn(x, rep);
  return __fsub_rn(x, __fadd_rn(__fmul_rn(static_cast<float>(count), freq), pres));
}

// Philox4x32-10 (Salmon et al., SC'11), first output word.  Key = seed halves; counter words =
// (position lo, position hi, draw counter lo, draw counter hi).
__device__ __forceinline__ uint32_t philox_word0(uint64_t seed, uint64_t pos, uint64_t ctr) {
  uint32_t c0 = static_cast<uint32_t>(pos), c1 = static_cast<uint32_t>(pos >> 32);
  uint32_t c2 = static_cast<uint32_t>(ctr), c3 = static_cast<uint32_t>(ctr >> 32);
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo_a = 0xD2511F53u * c0, hi_a = __umulhi(0xD2511F53u, c0);
    const uint32_t lo_b = 0xCD9E8D57u * c2, hi_b = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi_b ^ c1 ^ k0;
    const uint32_t n2 = hi_a ^ c3 ^ k1;
    c0 = n0;
    c1 = lo_b;
    c2 = n2;
    c3 = lo_a;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c0;
}

// Online (max, sum of exp(x - max)) pair, base-2 exponent with log2(e) folded in.
constexpr float LOG2E = 1.4426950408889634f;

struct MaxSum {
  float m, s;
};

__device__ __forceinline__ MaxSum ms_combine(MaxSum a, MaxSum b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return {M, 0.0f};
  const float sa = (a.m == -INFINITY) ? 0.0f : a.s * ex2_approx((a.m - M) * LOG2E);
  const float sb = (b.m == -INFINITY) ? 0.0f : b.s * ex2_approx((b.m - M) * LOG2E);
  return {M, sa + sb};
}

__device__ __forceinline__ MaxSum warp_ms(MaxSum x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    MaxSum y{__shfl_xor_sync(FULL_MASK, x.m, off), __shfl_xor_sync(FULL_MASK, x.s, off)};
    x = ms_combine(x, y);
  }
  return x;
}

// Warp (max, sum of exp) of per-lane pairs: the max by one redux on order keys, then every
// lane's sum rescaled to it and added by butterfly shuffles (short dependency chain).
__device__ __forceinline__ MaxSum warp_ms_fast(MaxSum x) {
  const uint32_t km = __reduce_max_sync(FULL_MASK, order_key(x.m));
  const float M = (km == 0u) ? -INFINITY : key_value(km);
  float s = (x.m == -INFINITY || M == -INFINITY || !(x.s > 0.0f)) ? 0.0f : x.s * ex2_approx((x.m - M) * LOG2E);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(FULL_MASK, s, off);
  return {M, s};
}

// ------------------------------------------------------------------------------ double-word fp32
// A value carried as an unevaluated sum hi + lo of two floats, added with Knuth's TwoSum (an
// error-free transformation), so a prefix sum of <= 64 terms keeps ~44 significant bits without
// FP64 arithmetic.
struct DW {
  float hi, lo;
};

__device__ __forceinline__ DW two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

__device__ __forceinline__ DW dw_add(DW x, DW y) {
  const DW s = two_sum(x.hi, y.hi);
  const float lo = __fadd_rn(__fadd_rn(x.lo, y.lo), s.lo);
  const float hi = __fadd_rn(s.hi, lo);
  return {hi, __fsub_rn(lo, __fsub_rn(hi, s.hi))};
}

// x * y for a float y, with the product's rounding error recovered by a fused multiply-add.
__device__ __forceinline__ DW dw_mul_f(DW x, float y) {
  const float p = __fmul_rn(x.hi, y);
  const float e = __fmaf_rn(x.hi, y, -p);
  const float lo = __fadd_rn(e, __fmul_rn(x.lo, y));
  const float hi = __fadd_rn(p, lo);
  return {hi, __fsub_rn(lo, __fsub_rn(hi, p))};
}

// Sign of a - b for double-word values (the high parts are close whenever the sign is in doubt).
__device__ __forceinline__ bool dw_less(DW a, DW b) {
  return __fadd_rn(__fsub_rn(a.hi, b.hi), __fsub_rn(a.lo, b.lo)) < 0.0f;
}

__device__ __forceinline__ DW warp_scan_dw(DW x, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const DW y{__shfl_up_sync(FULL_MASK, x.hi, off), __shfl_up_sync(FULL_MASK, x.lo, off)};
    if (lane >= off) x = dw_add(y, x);
  }
  return x;
}

__device__ __forceinline__ DW shfl_dw(DW x, int src) {
  return {__shfl_sync(FULL_MASK, x.hi, src), __shfl_sync(FULL_MASK, x.lo, src)};
}

__device__ __forceinline__ float warp_scan_f(float x, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(FULL_MASK, x, off);
    if (lane >= off) x += y;
  }
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(FULL_MASK, x, off);
  return x;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t y = __shfl_xor_sync(FULL_MASK, x, off);
    x = (y > x) ? y : x;
  }
  return x;
}

}  // namespace strata
