// cider_device.cuh -- device helpers shared by the sm_103a kernels: inline PTX
// for mbarriers, TMA bulk-tensor loads and the tcgen05 tensor-core / tensor
// memory instructions, bounded waits, and the exact integer -> fp16
// conversions that feed integer operands to the fp16 tensor pipe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace cider {

// Error bits written to the library's device error word.
constexpr int kDevErrTimeout = 1;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Barrier over `count` threads (a multiple of 32) of the CTA, with id 1..15.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// 16-byte shared-memory store to a 32-bit shared address.
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint32_t (&v)[4]) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3])
               : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
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

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_wait_bounded, but polling with the non-blocking test_wait (the
// thread never suspends): for short waits on data that is almost there.
__device__ __forceinline__ bool mbar_spin_bounded(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t* abort_flag, int* err,
                                                  uint64_t timeout_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint64_t n = 1;; ++n) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((n & 255) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        *abort_flag = 1u;
        atomicOr(err, kDevErrTimeout);
        return false;
      }
    }
  }
}

// Bounded wait for the phase with the given parity.  Gives up when another
// thread of the CTA raised `abort_flag`, after `max_polls` polls (0 = no poll
// limit), or after `timeout_ns` of global time; a give-up of its own sets
// `abort_flag` and the device error word.  Returns true when the phase
// completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t* abort_flag, int* err,
                                                  uint64_t timeout_ns, uint64_t max_polls = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint64_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    bool give_up = (max_polls != 0 && n >= max_polls);
    if (!give_up && (n & 63) == 0) give_up = (global_timer_ns() - t0) > timeout_ns;
    if (give_up) {
      *abort_flag = 1u;
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// As mbar_wait_bounded, but each poll suspends the thread in hardware until
// the phase completes or about `hint_ns` pass, so that waiting warps leave
// the issue slots to the warps doing work (in kernels with many more waiting
// warps than working ones).
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_sleep_bounded(uint32_t bar, uint32_t parity,
                                                   volatile uint32_t* abort_flag, int* err,
                                                   uint64_t timeout_ns) {
  if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort_flag = 1u;
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// ------------------------------------------------- flags in global memory
// A counter that other CTAs of the same launch wait on.  Every thread that
// wrote data the waiters will read adds 1 with release semantics (covering
// its own earlier stores); a waiter that reads the full count with acquire
// semantics then sees every one of those stores.
__device__ __forceinline__ void gpu_count_release(int* counter) {
  asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(counter) : "memory");
}

__device__ __forceinline__ int gpu_load_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *counter >= target (same give-up rules as
// mbar_wait_bounded).
__device__ __forceinline__ bool gpu_count_wait_bounded(const int* counter, int target,
                                                       volatile uint32_t* abort_flag, int* err,
                                                       uint64_t timeout_ns) {
  if (gpu_load_acquire(counter) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint64_t n = 1;; ++n) {
    __nanosleep(64);
    if (gpu_load_acquire(counter) >= target) return true;
    if (*abort_flag) return false;
    if ((n & 15) == 0 && global_timer_ns() - t0 > timeout_ns) {
      *abort_flag = 1u;
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------- clusters
// Rank of this CTA in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Barrier over every thread of every CTA of the cluster (all threads of each
// warp must execute it), with release / acquire ordering at cluster scope.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier anywhere in the cluster (address from mapa_shared),
// with the default (CTA-scope release) semantics.  Shared-memory operands
// written by this thread for the tensor core are published with
// fence_proxy_async_smem() before the arrive; a cluster-scope release here
// would cost ~1500 cycles per arrive on GB300 and serialise the pipeline.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Tiled shared -> global copy by the TMA engine (box of the tensor map, from
// a box-shaped, swizzled shared-memory tile); parts of the box outside the
// tensor are not written.  Completion is tracked by bulk async-groups of the
// issuing thread (bulk_commit_group / bulk_wait_group*).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until at most N of this thread's bulk groups are still reading their shared-memory sources.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Until at most N of this thread's bulk groups are incomplete (writes included).
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// As tma_load_2d, issued by either CTA of a CTA pair into its own shared
// memory, with the completion counted on `bar` (a shared::cluster address,
// which may be in the peer CTA).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Contiguous global -> shared copy by the TMA engine, completing `bytes` of
// transaction count on `bar`.  Addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it on the stream still
// runs; pdl_wait() returns once that kernel has completed and its writes are
// visible (at once when the launch had no such attribute).  The kernel before
// lets its dependents start early with pdl_launch_dependents().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// CTA-pair (cta_group::2) forms.  One warp of EACH CTA of the pair executes
// the allocation / deallocation; the allocation holds the same columns in
// both CTAs' tensor memories.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// Arrive on the mbarrier at the same shared-memory offset in every CTA of
// `cta_mask` once all prior tcgen05 operations of this thread completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
// D (+)= A * B^T on a CTA pair, kind::f16, both operands in shared memory:
// A rows [0, M/2) from this CTA and [M/2, M) from the peer, at the same
// offset; B column j from the CTA j / (N/2), row j % (N/2); D rows of each
// CTA in its own tensor memory, all N columns.  Issued by one thread of the
// pair's even CTA.
__device__ __forceinline__ void tc_mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, one CTA.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, one CTA.
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp reads lane
// (lane field of taddr) + t; register i holds column (column of taddr) + i.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address, 16-byte units
  d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2u) << 61;                 // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (both K-major), fp32 D,
// shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (0u << 7) | (0u << 10)                    // A, B format: f16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// ---------------------------------------------------------------- loads
// Asynchronous 4-byte global -> shared copy (completion tracked per thread by
// commit groups); `valid` false writes zero and reads nothing.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's most recent commit groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------- outputs
// The bits of one output value: the fp32 result rounded once to fp16 or to
// bf16 (round to nearest even either way).
template <bool BF16>
__device__ __forceinline__ uint16_t y_bits(float v) {
  if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}
// Two outputs at once, low | high << 16: one paired conversion instruction,
// each value rounded to nearest even exactly as y_bits does.
template <bool BF16>
__device__ __forceinline__ uint32_t y_bits2(float lo, float hi) {
  uint32_t u;
  if constexpr (BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    memcpy(&u, &h, 4);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    memcpy(&u, &h, 4);
  }
  return u;
}


// ---------------------------------------------------------------- exact integer -> fp16
// Four int8 codes (byte i = code i) -> half2 {c0, c1} and {c2, c3}, exactly.
// The byte is moved to offset binary (code + 128) and placed in the mantissa
// of 1024.0 (exponent with unit spacing), giving 1024 + code + 128; then
// 1152 is subtracted.  Every intermediate is an integer below 2048, exact in
// fp16.
__device__ __forceinline__ void s8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x64646464u, 0x5140u);
  uint32_t b = __byte_perm(u, 0x64646464u, 0x7362u);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// Eight packed INT4 codes (byte j: element 2j low nibble, 2j+1 high nibble,
// two's complement) -> four half2 {e0,e1} {e2,e3} {e4,e5} {e6,e7}, exactly.
// Nibbles go to offset binary t = code + 8; for each byte the low nibble is
// placed in the mantissa of 1024.0 (1024 + t) and the high nibble four bits
// up (1024 + 16 t); one fp16 FMA per pair then gives (t - 8) for both:
// (1024 + t) * 1 - 1032 and (1024 + 16 t) / 16 - 72.  All exact.
__device__ __forceinline__ void s4x8_to_h2x4(uint32_t w, uint32_t (&h)[4]) {
  const uint32_t u = w ^ 0x88888888u;
  const __half2 scale = __halves2half2(__ushort_as_half(0x3C00u), __ushort_as_half(0x2C00u));
  const __half2 bias = __halves2half2(__ushort_as_half(0xE408u), __ushort_as_half(0xD480u));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t sel = 0x4040u | (static_cast<uint32_t>(j) << 8) | static_cast<uint32_t>(j);
    uint32_t x = (__byte_perm(u, 0u, sel) & 0x00F0000Fu) | 0x64006400u;
    __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), scale, bias);
    h[j] = *reinterpret_cast<uint32_t*>(&r);
  }
}

// The same eight codes as fp16 pairs of even and of odd codes:
// even = {c0, c2} {c4, c6}, odd = {c1, c3} {c5, c7} (the order in which
// offset_nibbles_to_s8x4 of the low / high nibbles followed by s8x4_to_h2x2
// gives them), in one step: bytes (0, 1) and (2, 3) go to the two halves,
// the low nibbles into the mantissa of 1024 (1024 + t, minus 1032) and the
// high nibbles four bits up (1024 + 16 t, times 1/16 minus 72).  All exact.
__device__ __forceinline__ void s4x8_to_h2_eo(uint32_t w, uint32_t (&ev)[2], uint32_t (&od)[2]) {
  const uint32_t u = w ^ 0x88888888u;
  const __half2 one = __halves2half2(__ushort_as_half(0x3C00u), __ushort_as_half(0x3C00u));
  const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00u), __ushort_as_half(0x2C00u));
  const __half2 bias_lo = __halves2half2(__ushort_as_half(0xE408u), __ushort_as_half(0xE408u));
  const __half2 bias_hi = __halves2half2(__ushort_as_half(0xD480u), __ushort_as_half(0xD480u));
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const uint32_t b = __byte_perm(u, 0u, p == 0 ? 0x4140u : 0x4342u);   // [byte 2p, 0, byte 2p+1, 0]
    uint32_t lo = (b & 0x000F000Fu) | 0x64006400u;
    uint32_t hi = (b & 0x00F000F0u) | 0x64006400u;
    const __half2 rl = __hfma2(*reinterpret_cast<__half2*>(&lo), one, bias_lo);
    const __half2 rh = __hfma2(*reinterpret_cast<__half2*>(&hi), sixteenth, bias_hi);
    ev[p] = *reinterpret_cast<const uint32_t*>(&rl);
    od[p] = *reinterpret_cast<const uint32_t*>(&rh);
  }
}

// Eight int8 codes in natural order (lo: codes 0..3, hi: codes 4..7) as
// fp16 pairs of even codes {c0, c2} {c4, c6} and of odd codes {c1, c3}
// {c5, c7}, exactly: the byte permutes that place each code in the mantissa
// of 1024 (offset binary, code + 128; minus 1152) also pick the even / odd codes.
__device__ __forceinline__ void s8x8_to_h2_eo(uint32_t lo, uint32_t hi, uint32_t (&ev)[2],
                                              uint32_t (&od)[2]) {
  const uint32_t l = lo ^ 0x80808080u, h = hi ^ 0x80808080u;
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
  uint32_t r[4] = {__byte_perm(l, 0x64646464u, 0x5240u), __byte_perm(h, 0x64646464u, 0x5240u),
                   __byte_perm(l, 0x64646464u, 0x5341u), __byte_perm(h, 0x64646464u, 0x5341u)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 v = __hsub2(*reinterpret_cast<__half2*>(&r[i]), bias);
    r[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  ev[0] = r[0];
  ev[1] = r[1];
  od[0] = r[2];
  od[1] = r[3];
}

// x / s correctly rounded (IEEE binary32, round to nearest even), from
// r = RN(1/s) and two FMAs: q0 = RN(x r) is within one ulp of x / s, the
// residual x - s q0 is exact in one FMA, and RN(q0 + residual * r) is the
// correctly rounded quotient (Markstein's theorem; P. Markstein, "IA-64 and
// Elementary Functions", 2000; J.-M. Muller et al., "Handbook of
// Floating-Point Arithmetic", division by FMA).  The theorem needs no
// overflow or underflow on the way, which holds here: |x / s| <= 127 and the
// residual is at least 2^-24 |s q0| whenever it is not zero.
__device__ __forceinline__ float div_rn_by(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q0, s, x);
  return __fmaf_rn(e, r, q0);
}

// Symmetric INT8 code of x for scale s (r = RN(1/s)): clamp(rint(x / s), +-127).
__device__ __forceinline__ float act_code(float x, float s, float r) {
  const float q = rintf(div_rn_by(x, s, r));
  return fminf(fmaxf(q, -127.0f), 127.0f);
}

// Four INT4 codes in the low nibbles of the bytes of t (high nibbles zero),
// as offset binary (code + 8) -> four sign-correct int8 codes, carry-free:
// (t + 0x78) ^ 0x80 maps 0..7 -> -8..-1 and 8..15 -> 0..7 in every byte.
__device__ __forceinline__ uint32_t offset_nibbles_to_s8x4(uint32_t t) {
  return (t + 0x78787878u) ^ 0x80808080u;
}

}  // namespace cider
