// Device helpers shared by the sm_103a kernels: mbarriers with bounded waits,
// TMA tile loads, tcgen05 (MMA, TMEM load/store/alloc), cluster barriers and
// distributed shared memory. Inline PTX only; no third-party headers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace mla {

// Device error word of this translation unit (each kernel file has its own),
// read and cleared by mla_check_device_errors.
static __device__ uint32_t g_device_error;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void flag_error(uint32_t bits) { atomicOr(&g_device_error, bits); }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
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
// Test the phase; if it is not complete the thread is suspended in hardware
// until it completes or about `hint_ns` pass, so waiting warps do not take
// issue slots from the warps doing work.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 1000000u) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Limit of the waits that let copies / MMAs already in flight finish before a
// CTA that gave up leaves (they always complete; this only bounds the wait).
constexpr uint64_t kDrainTimeoutNs = 2000000000ull;

// Suspend-time hint of the waits: at most 1 ms, and no longer than the
// wait's own limit, so a short limit is checked about that often.
__device__ __forceinline__ uint32_t wait_hint_ns(uint64_t timeout_ns) {
  return timeout_ns < 1000000ull ? static_cast<uint32_t>(timeout_ns) : 1000000u;
}

// Wait for the phase with the given parity to complete. Gives up after
// `timeout_ns` of wall time, flags MLA_DEVERR_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint32_t hint = wait_hint_ns(timeout_ns);
  if (__builtin_expect(mbar_try_wait(bar, parity, hint), 1)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity, hint)) return true;
    if (globaltimer_ns() - t0 > timeout_ns) {
      flag_error(MLA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (tensor tile loads into shared memory, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Prefetch `bytes` contiguous bytes into L2 (address and size multiples of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// 2D tile load: box origin (x = innermost element index, y = row).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 4D tile load (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            int32_t c3, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Prefetch a 2D tile into L2 (no shared-memory destination, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Arrive on a named barrier without waiting (the consumer side calls named_bar_sync).
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads:
// every thread gets the same answer (a uniform decision, e.g. to abort).
__device__ __forceinline__ bool named_bar_sync_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

// ---------------------------------------------------------------------------
// Thread-block cluster and distributed shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split cluster barrier: arrive (release) now, wait (acquire) later. Every
// thread that arrives must wait before it arrives again.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// Arrival with no memory ordering: for a barrier that only has to keep a CTA until its peers have
// reached a point (their shared-memory traffic to it already observed complete on mbarriers).
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }
// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}
// Loads from another CTA's shared memory. Only used on data published before
// a cluster barrier, so they carry no ordering of their own and can overlap.
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 dsmem_ld_f32x4(uint32_t addr) {
  float4 v;
  asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// Plain 32-bit store to another CTA's shared memory (address from dsmem_addr);
// ordered before a following cluster barrier's release.
__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// After an abort: spin for `ns` nanoseconds, so that copies and remote stores
// already issued between the CTAs of a cluster complete before a CTA exits.
__device__ __forceinline__ void settle_in_flight(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) {
  }
}
// Asynchronous 16-byte store to another CTA's shared memory; its bytes count
// as completed transactions on that CTA's mbarrier `remote_bar` (both
// addresses from dsmem_addr). The sender does not wait for it.
__device__ __forceinline__ void dsmem_st_async_f32x4(uint32_t addr, float4 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
               : "memory");
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from this
// CTA's shared memory to another CTA's (dst and remote_bar from dsmem_addr); the
// bytes complete transactions on that CTA's mbarrier. Reads of the source are
// finished once that mbarrier's phase completes.
__device__ __forceinline__ void dsmem_bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t remote_bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst),
               "r"(smem_u32(src)), "r"(bytes), "r"(remote_bar)
               : "memory");
}
// 16-byte global -> shared copy, zero-filled past `src_bytes` (0 or 16); completes at cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// Arrive without memory ordering on an mbarrier of another CTA: a pure signal,
// for use only where every access it must follow has completed (values
// consumed and a CTA barrier passed since).
__device__ __forceinline__ void mbar_remote_arrive_relaxed(uint32_t addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// Bounded wait on a local mbarrier whose arrivals come from other CTAs of the
// cluster: acquire at cluster scope, so their stores before the arrive are visible.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint32_t hint = wait_hint_ns(timeout_ns);
  auto test = [&]() -> bool {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint)
        : "memory");
    return ok != 0;
  };
  if (__builtin_expect(test(), 1)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (test()) return true;
    if (globaltimer_ns() - t0 > timeout_ns) {
      flag_error(MLA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ---------------------------------------------------------------------------
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
// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]; A is M x K with row m in TMEM lane m and K packed
// two 16-bit elements per 32-bit column (8 columns per K=16 step).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// A shared-memory matrix descriptor as its two 32-bit halves. The start
// address field (address / 16) is in the low half, and an offset inside one
// CTA's shared memory never carries out of it, so advancing a descriptor is a
// single 32-bit add. The MMA issue loops use this form: per instruction they
// do one add per operand, so back-to-back MMAs keep the tensor core busy
// (64-bit descriptor arithmetic between them left it idle about half the time).
struct Desc2 {
  uint32_t lo, hi;
};
__device__ __forceinline__ Desc2 desc2(uint64_t d) {
  return Desc2{static_cast<uint32_t>(d), static_cast<uint32_t>(d >> 32)};
}
// The descriptor advanced by `bytes` (a multiple of 16).
__device__ __forceinline__ Desc2 desc2_add(Desc2 d, uint32_t bytes) { return Desc2{d.lo + (bytes >> 4), d.hi}; }
// D[tmem] (+)= A[smem] * B[smem]; a and b advanced by a16 / b16 units of 16 bytes.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, Desc2 a, uint32_t a16, Desc2 b, uint32_t b16, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 da, db;\n setp.ne.b32 p, %6, 0;\n mov.b64 da, {%1, %2};\n"
      " mov.b64 db, {%3, %4};\n tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n}\n" ::"r"(d_tmem),
      "r"(a.lo + a16), "r"(a.hi), "r"(b.lo + b16), "r"(b.hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// Arrive on the mbarrier at `bar`'s offset in every CTA of the cluster whose
// rank bit is set in `cta_mask`, once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Warp loads / stores 32 lanes x 8 consecutive 32-bit columns (lane = thread).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
// Warp loads 32 lanes x 16 consecutive 32-bit columns (lane = thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
// start/lbo/sbo in bytes; the fixed "version" field (bits 46-47) is 1.
// K-major operands: sbo = stride between 8-row groups (lbo unused).
// MN-major operands: lbo = stride between 64-element MN blocks, sbo = stride
// between 8-row K groups.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t start, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((start >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;  // SWIZZLE_128B
  return d;
}

// The same for a K-major operand whose rows are 64 bytes (two K=16 steps of
// 16-bit elements) stored with the 64-byte swizzle (16-byte chunk c of row r
// at position c ^ ((r / 2) % 4), as a TMA box with CU_TENSOR_MAP_SWIZZLE_64B
// lands): sbo = stride between 8-row groups (512 B when the rows are packed);
// the second K step starts 32 bytes in.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t start, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((start >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;  // leading byte offset: unused within one swizzle atom
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(4) << 61;  // SWIZZLE_64B
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with an fp32 accumulator.
// a_mn / b_mn: operand stored MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool bf16, bool a_mn, bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of element (row, col) inside a [rows x 64] 16-bit tile stored
// with the 128-byte swizzle (rows of 128 bytes; the 16-byte chunk index is
// XORed with row % 8). The tile base must be 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col) {
  return row * 128u + ((((col >> 3) ^ row) & 7u) << 4) + ((col & 7u) << 1);
}

// Byte offset of 16-bit element (row, col) in rows of 64 bytes stored with the
// 64-byte swizzle (the layout smem_desc_sw64 describes).
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t col) {
  return row * 64u + ((((col >> 3) ^ (row >> 1)) & 3u) << 4) + ((col & 7u) << 1);
}

// ---------------------------------------------------------------------------
// 16-bit conversions
// ---------------------------------------------------------------------------
template <bool BF16>
__device__ __forceinline__ float h2f(uint16_t v) {
  if constexpr (BF16) {
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  } else {
    return __half2float(__ushort_as_half(v));
  }
}
// Programmatic dependent launch. A grid that calls pdl_launch_dependents lets the
// next kernel of its stream, when that one is launched with programmatic stream
// serialization, start before this grid ends; the dependent must call pdl_wait
// before it touches memory this grid writes: the wait returns once every
// prerequisite grid has completed and its writes are visible. Without the
// launch attribute both are no-ops in effect (the dependent starts after the end).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// below 2^-22 per the PTX ISA); 2^-inf = +0, so masked scores need no test.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <bool BF16>
__device__ __forceinline__ uint16_t f2h(float v) {
  if constexpr (BF16) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  } else {
    return __half_as_ushort(__float2half_rn(v));
  }
}

// Ticket for "the last one merges": an add with acquire-release semantics at device scope. It
// releases what this thread has written, and what other threads wrote before a barrier this
// thread has passed, before the count moves; the thread that reads the final count acquires
// what the others released with their own adds.
__device__ __forceinline__ uint32_t ticket_add_acq_rel(uint32_t* t) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
  return old;
}
// Reset a ticket for the next call: nothing else touches it until this grid has completed.
__device__ __forceinline__ void ticket_reset(uint32_t* t) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(t) : "memory");
}
// ---------------------------------------------------------------------------
// Work of one CTA: request, chunk bounds, output slot, token sub-range.
// ---------------------------------------------------------------------------
struct CtaWork {
  int32_t b, t0, t1, slot;  // chunk
  int32_t L;                // context length of request b
  int32_t sub0, sub1;       // this CTA's tokens [sub0, sub1)
  int32_t row0, nrows;      // query rows [row0, row0 + nrows) of this CTA
};

// Chunk rule shared with the planner: C = ceil(ceil(L/P)/bs)*bs.
__device__ __forceinline__ void uniform_chunk(int32_t L, int32_t P, int32_t p, int32_t bs, int32_t* t0,
                                              int32_t* t1) {
  int32_t per = (L + P - 1) / P;
  int32_t C = ((per + bs - 1) / bs) * bs;
  if (C < bs) C = bs;
  long long a = static_cast<long long>(p) * C, e = static_cast<long long>(p + 1) * C;
  *t0 = static_cast<int32_t>(a < L ? a : L);
  *t1 = static_cast<int32_t>(e < L ? e : L);
}

// Fill the chunk (blockIdx.y, or `chunk`), the CTA's token sub-range (runs of
// `unit`-token tiles split evenly over the cluster, or over `nparts` groups,
// this CTA in group `part`) and its query rows (row group blockIdx.z, or
// `row_group`). Tokens are trimmed to the last one any row
// of this CTA can see under the causal rule.
__device__ __forceinline__ CtaWork cta_work(const PartialParams& p, int32_t rows_per_cta,
                                            int32_t unit = kTileTokens, int32_t part = -1, int32_t nparts = 0,
                                            int32_t chunk = -1, int32_t row_group = -1) {
  CtaWork w;
  const int32_t n = (chunk >= 0) ? chunk : static_cast<int32_t>(blockIdx.y);
  if (p.chunks != nullptr) {
    const int4 c = reinterpret_cast<const int4*>(p.chunks)[n];
    w.b = c.x;
    w.t0 = c.y;
    w.t1 = c.z;
    w.slot = c.w;
  } else {
    w.b = n / p.num_parts;
    w.slot = n;
    w.t0 = 0;
    w.t1 = 0;
  }
  w.L = 0;
  if (w.b >= 0 && w.b < p.B) w.L = p.context_lens[w.b];
  if (w.L < 0) w.L = 0;
  if (p.chunks == nullptr) uniform_chunk(w.L, p.num_parts, n % p.num_parts, p.bs, &w.t0, &w.t1);
  if (w.t1 > w.L) w.t1 = w.L;
  if (w.t0 < 0) w.t0 = 0;
  if (w.t0 > w.t1) w.t0 = w.t1;
  w.row0 = ((row_group >= 0) ? row_group : static_cast<int32_t>(blockIdx.z)) * rows_per_cta;
  const int32_t total_rows = p.q_len * p.H;
  w.nrows = total_rows - w.row0;
  if (w.nrows > rows_per_cta) w.nrows = rows_per_cta;
  if (w.nrows < 0) w.nrows = 0;
  int32_t tend = w.t1;
  if (p.causal && w.nrows > 0) {
    const int32_t i_last = (w.row0 + w.nrows - 1) / p.H;
    const int32_t lim = w.L - p.q_len + i_last + 1;  // exclusive bound of visible tokens
    if (tend > lim) tend = lim;
    if (tend < w.t0) tend = w.t0;
  }
  const int32_t units = (tend - w.t0 + unit - 1) / unit;
  const int32_t C = (nparts > 0) ? nparts : static_cast<int32_t>(cluster_nctarank());
  const int32_t k = (nparts > 0) ? part : static_cast<int32_t>(cluster_ctarank());
  const int32_t u0 = static_cast<int32_t>((static_cast<long long>(units) * k) / C);
  const int32_t u1 = static_cast<int32_t>((static_cast<long long>(units) * (k + 1)) / C);
  w.sub0 = w.t0 + u0 * unit;
  w.sub1 = w.t0 + u1 * unit;
  if (w.sub1 > tend) w.sub1 = tend;
  if (w.sub0 > w.sub1) w.sub0 = w.sub1;
  return w;
}

// Page id of logical page `pg` of request b, with a range check: an entry
// outside [0, num_blocks) is flagged and mapped to -1 (TMA then reads zeros).
__device__ __forceinline__ int32_t checked_page(const PartialParams& p, int32_t b, int32_t pg) {
  int32_t pid = __ldg(p.block_table + static_cast<long long>(b) * p.max_blocks + pg);
  if (pid < 0 || pid >= p.num_blocks) {
    flag_error(MLA_DEVERR_BAD_PAGE);
    pid = -1;
  }
  return pid;
}

// Combine the (max, sum, O) staged by the CTAs of this cluster: this CTA
// writes columns [rank*512/C, (rank+1)*512/C) of each of its rows, rank 0
// also the LSE. Fixed rank order, so the result is bitwise reproducible.
// `ostage` is [rows][512] fp32, `mst`/`lst` [rows] fp32, same offsets in every
// CTA. The per-rank loads are independent (unrolled over the 16 possible ranks).
// The result goes to slot `dst_slot` of `dst_partials` / `dst_lse` (the chunk's
// own slot, or a sub-partial slot of the workspace).
__device__ __forceinline__ void cluster_combine_to(const PartialParams& p, const CtaWork& w, const float* ostage,
                                                   const float* mst, const float* lst, int tid, int nthreads,
                                                   float* dst_partials, float* dst_lse, long long dst_slot) {
  const int rows_total = p.q_len * p.H;
  const uint32_t C = cluster_nctarank(), kr = cluster_ctarank();
  const int dcols = kRank / static_cast<int>(C);
  const int dbeg = static_cast<int>(kr) * dcols;
  const int n4 = dcols / 4;
  const int items = w.nrows * n4 + ((kr == 0) ? w.nrows : 0);  // column groups, then LSE rows
  for (int idx = tid; idx < items; idx += nthreads) {
    const bool is_lse = idx >= w.nrows * n4;
    const int r = is_lse ? idx - w.nrows * n4 : idx / n4;
    const int d = is_lse ? 0 : dbeg + (idx % n4) * 4;
    float mj[16], wj[16];
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      mj[j] = (j < static_cast<int>(C)) ? dsmem_ld_f32(dsmem_addr(mst + r, j)) : -INFINITY;
      M = fmaxf(M, mj[j]);
    }
    float den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int j = 0; j < 16; ++j) wj[j] = (mj[j] == -INFINITY) ? 0.f : exp2f(mj[j] - M);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (j < static_cast<int>(C)) {
          den = fmaf(wj[j], dsmem_ld_f32(dsmem_addr(lst + r, j)), den);
          if (!is_lse) {
            const float4 v = dsmem_ld_f32x4(dsmem_addr(ostage + r * kRank + d, j));
            num.x = fmaf(wj[j], v.x, num.x);
            num.y = fmaf(wj[j], v.y, num.y);
            num.z = fmaf(wj[j], v.z, num.z);
            num.w = fmaf(wj[j], v.w, num.w);
          }
        }
      }
    }
    if (is_lse) {
      dst_lse[dst_slot * rows_total + w.row0 + r] = (M == -INFINITY) ? -INFINITY : M + log2f(den);
    } else {
      float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) out = make_float4(num.x / den, num.y / den, num.z / den, num.w / den);
      const long long base = (dst_slot * rows_total + w.row0 + r) * kRank + d;
      *reinterpret_cast<float4*>(dst_partials + base) = out;
    }
  }
}
__device__ __forceinline__ void cluster_combine(const PartialParams& p, const CtaWork& w, const float* ostage,
                                                const float* mst, const float* lst, int tid, int nthreads) {
  cluster_combine_to(p, w, ostage, mst, lst, tid, nthreads, p.partials, p.lse, static_cast<long long>(w.slot));
}

// The merge of n partials (slots lo .. lo+n-1, normalized, base-2 LSE) for row r and the four
// columns [c, c + 4): the merge kernel's arithmetic in the merge kernel's order (the maximum LSE
// M, weights 2^(lse - M) with -inf giving 0, the weight sum and the fused multiply-adds in slot
// order, one division per column), so every merge built on it gives the bits mla_merge_states
// gives. Writes the normalized values (0 when every LSE is -inf), M and the weight sum.
// Partials and LSE written by other CTAs of the same grid are read through L2 (ld.global.cg).
__device__ __forceinline__ float4 merge_cols4(const float* partials, const float* lse_src, int lo, int n, int rows,
                                              int r, int c, bool values, float* M_out, float* den_out) {
  const long long stride = static_cast<long long>(rows) * kRank;  // one partial slot
  const float* lrow = lse_src + static_cast<long long>(lo) * rows + r;
  const float* vcol = partials + static_cast<long long>(lo) * stride + static_cast<long long>(r) * kRank + c;
  // the first 8 partials' LSE and values in one round of loads (the values do not depend on the
  // weights); further LSE in rounds of 8 for the maximum
  float l0[8];
  float4 v0[8];
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) {
    const bool in = jj < n;
    l0[jj] = in ? __ldcg(lrow + static_cast<long long>(jj) * rows) : -INFINITY;
    v0[jj] = (in && values) ? __ldcg(reinterpret_cast<const float4*>(vcol + jj * stride))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float M = -INFINITY;
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) M = fmaxf(M, l0[jj]);
  for (int j0 = 8; j0 < n; j0 += 8) {
    float lj[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) lj[jj] = (j0 + jj < n) ? __ldcg(lrow + static_cast<long long>(j0 + jj) * rows) : -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) M = fmaxf(M, lj[jj]);
  }
  float den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int j0 = 0; j0 < n; j0 += 8) {
      float lj[8];
      float4 v[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (j0 == 0) {
          lj[jj] = l0[jj];
          v[jj] = v0[jj];
        } else {
          const bool in = j0 + jj < n;
          lj[jj] = in ? __ldcg(lrow + static_cast<long long>(j0 + jj) * rows) : -INFINITY;
          v[jj] = (in && values) ? __ldcg(reinterpret_cast<const float4*>(vcol + (j0 + jj) * stride))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (j0 + jj < n) {
          const float wj = (lj[jj] == -INFINITY) ? 0.f : exp2f(lj[jj] - M);
          den += wj;
          acc.x = fmaf(wj, v[jj].x, acc.x);
          acc.y = fmaf(wj, v[jj].y, acc.y);
          acc.z = fmaf(wj, v[jj].z, acc.z);
          acc.w = fmaf(wj, v[jj].w, acc.w);
        }
      }
    }
    acc = make_float4(acc.x / den, acc.y / den, acc.z / den, acc.w / den);
  }
  *M_out = M;
  *den_out = den;
  return acc;
}

// The merged log2 LSE from merge_cols4's maximum and weight sum.
__device__ __forceinline__ float merged_lse(float M, float den) { return (M == -INFINITY) ? -INFINITY : M + log2f(den); }

// Four values rounded once to the output type (2: fp32, 1: bf16, 0: fp16) at element `off` of `out`.
__device__ __forceinline__ void store_out4(void* out, int32_t out_dtype, long long off, float4 acc) {
  if (out_dtype == 2) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + off) = acc;
    return;
  }
  const bool bf = (out_dtype == 1);
  const float f[4] = {acc.x, acc.y, acc.z, acc.w};
  uint16_t h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = bf ? f2h<true>(f[j]) : f2h<false>(f[j]);
  uint2 packed;
  packed.x = static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16);
  packed.y = static_cast<uint32_t>(h[2]) | (static_cast<uint32_t>(h[3]) << 16);
  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + off) = packed;
}

// Single-launch decode: the final merge of request b's chunk partials (slots lo .. hi-1) for
// columns [col0, col0 + ncols) of every row, into p.out (p.out_dtype) and, with write_lse,
// p.out_lse; the partials were written by other CTAs, ordered before this CTA's ticket by their
// fences.
__device__ __forceinline__ void request_merge(const PartialParams& p, int b, int lo, int hi, int col0, int ncols,
                                              bool write_lse, const float* lse_src, int tid, int nthreads) {
  const int rows = p.q_len * p.H;
  const int n4 = ncols / 4;
  const int items = rows * n4 + (write_lse ? rows : 0);
  for (int idx = tid; idx < items; idx += nthreads) {
    const bool is_lse = idx >= rows * n4;
    const int r = is_lse ? idx - rows * n4 : idx / n4;
    const int c = col0 + (is_lse ? 0 : (idx % n4) * 4);
    float M, den;
    const float4 acc = merge_cols4(p.partials, lse_src, lo, hi - lo, rows, r, c, !is_lse, &M, &den);
    const long long br = static_cast<long long>(b) * rows + r;
    if (is_lse) {
      if (p.out_lse != nullptr) p.out_lse[br] = merged_lse(M, den);
    } else {
      store_out4(p.out, p.out_dtype, br * kRank + c, acc);
    }
  }
}

// ---------------------------------------------------------------------------
// E4M3 caches: widening 8-bit tiles to fp16 in shared memory (the paired and
// the 128-row kernels)
// ---------------------------------------------------------------------------
// four E4M3 values (the bytes of w, lowest first) -> four fp16 values (two f16x2 words, lowest first);
// exact: every E4M3 value, its subnormals included, is an fp16 value
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  // volatile: kept between its step's load and stores, so the widening holds few values at a time
  asm volatile("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Shared-memory loads and stores of the in-place widening, as volatile asm without a memory clobber:
// kept in the order written (so a step's load can be issued ahead of earlier steps' stores, which the
// compiler could not prove independent), and ordered against the barrier operations around them
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, const uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

// 16 E4M3 bytes -> two 16-byte pieces of fp16 (bytes 0-7, bytes 8-15), stored at d0 and d1
__device__ __forceinline__ void widen16(const uint4 v, uint32_t d0, uint32_t d1) {
  uint4 a, b;
  e4m3x4_to_f16x4(v.x, a.x, a.y);
  e4m3x4_to_f16x4(v.y, a.z, a.w);
  e4m3x4_to_f16x4(v.z, b.x, b.y);
  e4m3x4_to_f16x4(v.w, b.z, b.w);
  sts128(d0, a);
  sts128(d1, b);
}

// One warp's steps of a widening part (three warps, two staged rows of 256 bytes a step: the CTA's half
// of the ckv columns of tokens t + 6 m and t + 6 m + 1, m < n), staged at stage_src + (t + 6 m) * 256;
// written to the 16-bit tile layout whose 8-token row groups of four swizzled [8 x 64] atoms are 4 KB
// apart. Each step's load is issued three steps ahead of its conversion.
__device__ __forceinline__ void widen_ckv_steps(uint32_t slot, uint32_t stage_src, int t, int n, int r2, int cbl,
                                                int kk) {
  if (n <= 0) return;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  uint4 b0 = lds128(stage_src + t * 256), b1 = z, b2 = z;
  if (n > 1) b1 = lds128(stage_src + (t + 6) * 256);
  if (n > 2) b2 = lds128(stage_src + (t + 12) * 256);
#pragma unroll 1
  for (int m = 0; m < n; ++m, t += 6) {
    const uint4 v = b0;
    b0 = b1;
    b1 = b2;
    if (m + 3 < n) b2 = lds128(stage_src + (t + 18) * 256);
    const int r = (t & 7) + r2;
    const uint32_t row = slot + (t >> 3) * 4096 + cbl * 1024 + r * 128;
    widen16(v, row + (((2 * kk) ^ r) << 4), row + (((2 * kk + 1) ^ r) << 4));
  }
}

// Request b's chunk slots [lo, hi): from the offsets, or the uniform split.
__device__ __forceinline__ void request_slots(const PartialParams& p, int b, int* lo, int* hi) {
  if (p.o_indptr != nullptr) {
    *lo = __ldg(p.o_indptr + b);
    *hi = __ldg(p.o_indptr + b + 1);
  } else {
    *lo = b * p.num_parts;
    *hi = (b + 1) * p.num_parts;
  }
}

}  // namespace mla
