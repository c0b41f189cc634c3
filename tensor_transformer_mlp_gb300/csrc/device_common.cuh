// Device-side helpers shared by the tpmlp kernels: inline-PTX wrappers for mbarriers,
// tensor-memory-access (TMA) copies and the 5th-generation tensor core (tcgen05),
// bounded waits, bf16 packing and the GeLU variants.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tpmlp_internal.h"

namespace tpmlp {

// ------------------------------------------------------------------ status / timing

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_timeout(unsigned int* status, unsigned int where) {
  if (status) atomicOr(status, kStatusTimeoutBit | (where << 8));
}

// ------------------------------------------------------------------ shared-memory addresses

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed, for at most limit_ns.
// Returns false (and records a timeout in *status) if the limit expired.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned int* status,
                                              unsigned int where, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  auto try_once = [&] { return mbar_try_wait(a, parity); };
  if (try_once()) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (try_once()) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      record_timeout(status, where);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* status,
                                          unsigned int where) {
  return mbar_wait_for(bar, parity, status, where, kWaitLimitNs);
}

// ------------------------------------------------------------------ CTA pairs (clusters of two)

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Every thread of every CTA in the cluster arrives, then waits for all the others.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (this CTA's or the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before its later async-proxy
// ones (a TMA load into a buffer the warp has just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled bulk copy global -> shared; completes `bytes` of transaction on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 2-D tiled copy into this CTA's shared memory whose completion is counted on an mbarrier that
// may sit in the peer CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

// tma_load_2d_pair with an L2 cache policy (l2_policy_evict_last).
__device__ __forceinline__ void tma_load_2d_pair_hint(void* dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                      int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// L2 cache policy for loads whose lines should outlive others' (evict_last).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 4-D tiled bulk copy global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0, int32_t c1,
                                            int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// 4-D tiled bulk copy shared -> global (the box's parts outside the tensor are not written),
// tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1,
                                             int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// 2-D tiled bulk copy shared -> global (the box's parts outside the tensor are not written),
// tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

// Brings a 2-D box of a tensor into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N of this thread's committed bulk groups still read their shared-memory
// source (the buffer of the others may be rewritten).
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until all of this thread's committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 1-D bulk copy global -> shared (addresses 16-byte aligned, size a multiple of 16);
// completes `bytes` of transaction on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05 (tensor memory + MMA)

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 x bf16 -> fp32, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Pair forms (cta_group::2): one allocation of ncols columns at the same address in both
// CTAs' tensor memory, made collectively by one warp of each CTA; likewise the release.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A * B across the pair: A's rows and B's columns split between the two CTAs' shared
// memory at the same offsets, D's rows split between their tensor memories. Issued by one
// thread of the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at this offset in every CTA of cta_mask when the pair MMAs
// issued so far have completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives lane (base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format, version 1) for a 128-byte-swizzled
// tile whose 8-row x 128-byte swizzle atoms start on 1024-byte boundaries.
//   lbo: byte distance between neighbouring atoms along the leading (contiguous) dimension
//   sbo: byte distance between neighbouring 8-row groups along the strided dimension
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)            // A major-ness (0 = K-major)
         | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// ------------------------------------------------------------------ numerics

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32); 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs: the sm_100-family f32x2 instructions (add, sub, mul, fma on two fp32 lanes,
// round to nearest) do two elements per issued instruction, with the same per-element rounding as
// the scalar forms.
struct F2 {
  unsigned long long v;
};
__device__ __forceinline__ F2 f2_make(float a, float b) {
  F2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_split(F2 a) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(a.v));
  return r;
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
  F2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
  F2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
  F2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}

constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kTanhC = 0.044715f;
constexpr float kInvSqrt2 = 0.7071067811865476f;
constexpr float kInvSqrt2Pi = 0.3989422804014327f;

// GeLU and its derivative in fp32. `precise` selects tanhf over the hardware tanh.approx.
// Tanh form with a = sqrt(2/pi), b = a * 0.044715: u = x (a + b x^2), phi = x/2 (1 + tanh u),
// phi' = (1 + tanh u) / 2 + x/2 (1 - tanh^2 u) (a + 3 b x^2); the fast path is arranged as
// FMAs (five FP operations and one tanh.approx for phi).
constexpr float kTanhA = kSqrt2OverPi;
constexpr float kTanhB = kSqrt2OverPi * kTanhC;

template <bool precise>
__device__ __forceinline__ float gelu_f(float x, int kind) {
  if (kind == kGeluErf) return 0.5f * x * (1.0f + erff(x * kInvSqrt2));
  if constexpr (precise) {
    const float u = kSqrt2OverPi * fmaf(kTanhC * x * x, x, x);
    return 0.5f * x * (1.0f + tanhf(u));
  } else {
    const float th = tanh_fast(x * fmaf(kTanhB, x * x, kTanhA));
    const float hx = 0.5f * x;
    return fmaf(hx, th, hx);
  }
}

template <bool precise>
__device__ __forceinline__ float gelu_grad_f(float x, int kind) {
  if (kind == kGeluErf) {
    const float cdf = 0.5f * (1.0f + erff(x * kInvSqrt2));
    return cdf + x * kInvSqrt2Pi * expf(-0.5f * x * x);
  }
  if constexpr (precise) {
    const float u = kSqrt2OverPi * fmaf(kTanhC * x * x, x, x);
    const float th = tanhf(u);
    return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * kSqrt2OverPi * fmaf(3.0f * kTanhC, x * x, 1.0f);
  } else {
    const float x2 = x * x;
    const float th = tanh_fast(x * fmaf(kTanhB, x2, kTanhA));
    const float dudx = fmaf(3.0f * kTanhB, x2, kTanhA);
    return fmaf(0.5f, th, 0.5f) + (0.5f * x * dudx) * fmaf(-th, th, 1.0f);
  }
}

// The tanh forms above on a pair of elements with f32x2 arithmetic (same operations and rounding
// per element as gelu_f<false> / gelu_grad_f<false>; tanh.approx per element).
__device__ __forceinline__ F2 tanh_fast2(F2 u) {
  const float2 v = f2_split(u);
  return f2_make(tanh_fast(v.x), tanh_fast(v.y));
}
__device__ __forceinline__ F2 gelu_tanh2(F2 x) {
  const F2 th = tanh_fast2(f2_mul(x, f2_fma(f2_make(kTanhB, kTanhB), f2_mul(x, x), f2_make(kTanhA, kTanhA))));
  const F2 hx = f2_mul(f2_make(0.5f, 0.5f), x);
  return f2_fma(hx, th, hx);
}
// phi' = (1 + th) / 2 + (x / 2) (a + 3 b x^2) (1 - th^2), arranged as
// fma((-x / 2) (a + 3 b x^2), th^2 - 1, fma(1/2, th, 1/2)).
__device__ __forceinline__ F2 gelu_grad_tanh2(F2 x) {
  const F2 x2 = f2_mul(x, x);
  const F2 th = tanh_fast2(f2_mul(x, f2_fma(f2_make(kTanhB, kTanhB), x2, f2_make(kTanhA, kTanhA))));
  const F2 dudx = f2_fma(f2_make(3.0f * kTanhB, 3.0f * kTanhB), x2, f2_make(kTanhA, kTanhA));
  const F2 p = f2_mul(f2_mul(f2_make(-0.5f, -0.5f), x), dudx);
  const F2 q = f2_fma(th, th, f2_make(-1.0f, -1.0f));
  return f2_fma(p, q, f2_fma(f2_make(0.5f, 0.5f), th, f2_make(0.5f, 0.5f)));
}


// Drop decision for one element: splitmix64(key) < threshold, with SplitMix64 as published by
// Steele, Lea and Flood (2014) / Vigna's splitmix64.c: add the golden-gamma increment, then the
// variant-13 mixer (xor-shift 30, multiply, xor-shift 27, multiply, xor-shift 31), mod 2^64.
constexpr uint64_t kSplitMixGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kSplitMixMul1 = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kSplitMixMul2 = 0x94D049BB133111EBull;

__host__ __device__ __forceinline__ bool hash_below(uint64_t key, uint64_t threshold) {
  uint64_t z = key + kSplitMixGamma;
  z = (z ^ (z >> 30)) * kSplitMixMul1;
  z = (z ^ (z >> 27)) * kSplitMixMul2;
  return (z ^ (z >> 31)) < threshold;
}

// drop_bits8 on keys whose shortcut below does not apply: eight full hashes.
static __host__ __device__ __noinline__ uint32_t drop_bits8_full(uint64_t base, uint64_t threshold) {
  uint32_t bits = 0;
  for (uint32_t e = 0; e < 8; ++e) bits |= (hash_below(base ^ e, threshold) ? 1u : 0u) << e;
  return bits;
}

// SplitMix64 of the eight keys base ^ e, e = 0..7, where base = seed ^ k0 with k0 a multiple of 8
// (so the keys are seed ^ (k0 + e)), with the work the eight keys share done once, in 32-bit
// halves:
//  * (base ^ e) + gamma = ((base & ~7) + gamma) + ((base & 7) ^ e), the last term in [0, 7].
//    Unless the low word of the first sum lies within 7 of 2^32, no key carries into the high
//    word, so the eight high words are equal, and so are the high word after the first
//    xor-shift and its share (high word x low word of the multiplier) of the first product.
//    If, in addition, adding the last term changes no key's bits 30 and 31 (the low word's low
//    30 bits are at most 2^30 - 8), the first xor-shift sends the same two bits down for every
//    key, so the word xor-ed into each key's low word is computed once too.
//  * The final xor-shift changes the high word only by flipping its bit 0 when its bit 31 is
//    set. For a threshold below 2^63 (p < 1/2) that changes neither "high word < threshold's
//    high word" nor equality with it, so high(e), the last product's high word, decides key e:
//    dropped iff high(e) < thi, unless high(e) == thi (probability 2^-32 per key), when only the
//    full hash decides.
// shortcut is false in the carry case, when a key changes bits 30-31 of the low word (each about
// one vector in 2^29), and for thresholds of 2^63 and above; a caller then uses hash_below (or
// drop_bits8_full) for all eight keys, and it does the same on a tie.
// kLow3 >= 0 promises base & 7 == kLow3 (the seed's low three bits), which makes each key's low
// word one addition of a constant.
template <int kLow3 = -1>
struct DropHash8 {
  uint32_t klo, low3, xs30, thi;
  uint64_t hi_product;
  bool shortcut;

  __host__ __device__ __forceinline__ DropHash8(uint64_t base, uint64_t threshold) {
    const uint64_t k = (base & ~7ull) + kSplitMixGamma;
    const uint32_t khi = static_cast<uint32_t>(k >> 32);
    klo = static_cast<uint32_t>(k);
    thi = static_cast<uint32_t>(threshold >> 32);
    shortcut = klo <= 0xFFFFFFF8u && (klo & 0x3FFFFFFFu) <= 0x3FFFFFF8u && thi < 0x80000000u;
    low3 = kLow3 >= 0 ? static_cast<uint32_t>(kLow3) : static_cast<uint32_t>(base) & 7u;
    // what the first xor-shift brings into every key's low word: the high word's low two bits
    // and the low word's own bits 30-31
    xs30 = (khi << 2) ^ (klo >> 30);
    hi_product = static_cast<uint64_t>((khi ^ (khi >> 30)) * static_cast<uint32_t>(kSplitMixMul1)) << 32;
  }

  __host__ __device__ __forceinline__ uint32_t high(uint32_t e) const {
    const uint32_t m1lo = static_cast<uint32_t>(kSplitMixMul1), m1hi = static_cast<uint32_t>(kSplitMixMul1 >> 32);
    const uint32_t m2lo = static_cast<uint32_t>(kSplitMixMul2), m2hi = static_cast<uint32_t>(kSplitMixMul2 >> 32);
    const uint32_t z0 = klo + (low3 ^ e);
    const uint32_t l1 = z0 ^ xs30;                                      // low word after xor-shift 30
    const uint64_t p1 = static_cast<uint64_t>(l1) * m1lo + hi_product;  // first product, minus l1 * m1hi
    const uint32_t a_lo = static_cast<uint32_t>(p1);
    const uint32_t a_hi = static_cast<uint32_t>(p1 >> 32) + l1 * m1hi;
    const uint32_t b_lo = a_lo ^ ((a_lo >> 27) | (a_hi << 5));         // xor-shift 27
    const uint32_t b_hi = a_hi ^ (a_hi >> 27);
    return static_cast<uint32_t>((static_cast<uint64_t>(b_lo) * m2lo) >> 32) + b_lo * m2hi + b_hi * m2lo;
  }
};

// The drop decisions of the eight keys base ^ e as bit e of the result (see DropHash8),
// identical to hash_below on each key.
template <int kLow3 = -1>
__host__ __device__ __forceinline__ uint32_t drop_bits8(uint64_t base, uint64_t threshold) {
  const DropHash8<kLow3> hs(base, threshold);
  if (!hs.shortcut) return drop_bits8_full(base, threshold);
  uint32_t bits = 0;
  bool tie = false;
#pragma unroll
  for (uint32_t e = 0; e < 8; ++e) {
    const uint32_t c = hs.high(e);
    bits |= (c < hs.thi ? 1u : 0u) << e;
    tie |= c == hs.thi;
  }
  return tie ? drop_bits8_full(base, threshold) : bits;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

}  // namespace tpmlp
