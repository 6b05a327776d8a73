// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tensor loads, and the tcgen05 tensor-core / tensor-memory instructions.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace h3 {

// Device error word: bit 0 = a pipeline wait ran out of time.  Read and
// cleared by h3dit_check_device_error().  The library is one translation
// unit (h3dit_api.cu includes every kernel file), so this is its only copy.
__device__ unsigned int g_device_error = 0;

constexpr unsigned int kErrTimeout = 1u;
// A legitimate wait in these kernels lasts microseconds; 2 s means the
// pipeline is stuck.  The limit lives in device memory so that a test can
// shorten it (h3dit_test_set_wait_limit) and watch a stalled pipeline give
// up within milliseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
__device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier
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
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The slow part of mbar_wait, out of line so that every wait site inlines
// only the single try-wait of the common case (this keeps the hot loops
// small: the attention kernel no longer spills).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort) {
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > g_wait_limit_ns) {
      *abort = 1;
      atomicOr(&g_device_error, kErrTimeout);
      return false;
    }
  }
}
// Wait until the phase of parity `parity` has completed.  Bounded: after
// g_wait_limit_ns (or once another role of the CTA gave up and raised *abort)
// it records the timeout and returns false so the caller can unwind.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort);
}

// Short bounded wait used only while unwinding after an abort.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 50000000ull) return;
  }
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Bulk (non-tensor) copy of `bytes` contiguous bytes from global memory into
// shared memory, completing on `bar`.  Both addresses 16-byte aligned, bytes
// a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Generic-proxy shared-memory writes made visible to the async proxy
// (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- launch overlap
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may be scheduled as the kernel before it on the stream
// retires its CTAs; it must call grid_dep_wait() before its first access to
// global memory, which returns once that kernel has completed and its
// writes are visible (so no earlier kernel still reads what it writes).
// Only shared-memory barrier setup, tensor-memory allocation and tensor-map
// prefetches (kernel parameters) come before it.  No kernel signals its
// dependents early (measured slower: the early CTAs crowd the running
// grid), so they are scheduled as its CTAs exit.  In a kernel launched
// without the attribute the wait is a no-op.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------- clusters
// Every thread of every CTA of the cluster; orders shared-memory writes
// before the barrier with reads (local or distributed) after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of `local` (a shared::cta address of this
// CTA's layout) in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float x, float y, float z, float w) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(x), "f"(y), "f"(z), "f"(w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float x) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(x) : "memory");
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ----------------------------------------------------------------- tcgen05
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
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
// tcgen05.commit from a whole converged warp: one elected lane commits.
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
      : "memory");
}
// True in exactly one lane of a converged warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile("{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n selp.u32 %0, 1, 0, e;\n}\n" : "=r"(r));
  return r != 0;
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// D(tmem) (+)= A(smem desc) * B(smem desc)^T, BF16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f16 with BF16 A/B, fp32 D, both operands
// K-major: D format bits [4,6) = 1, A format [7,10) = 1, B format [10,13) = 1,
// N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major operand stored in the 128-byte
// swizzle: rows of 128 bytes (64 BF16), 8-row core groups 1024 bytes apart,
// tile base 1024-byte aligned.  Start address bits [0,14) (>>4), leading
// offset [16,30) (unused for this layout), stride offset [32,46) (>>4),
// descriptor version 1 at bit 46, layout type 2 (128-byte swizzle) at [61,64).
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// The same descriptor split in two 32-bit words: the low word carries the
// start address (bits [0,14) = address >> 4) and the unused leading offset
// (1 at bit 16); the high word is the same for every operand of this layout
// (stride offset 1024 >> 4, version bit 46, 128-byte swizzle at [61,64)).
// Offsets inside an operand are added to the low word: shared-memory
// addresses stay below 2^18, so the 14-bit field never carries.
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr) { return ((saddr & 0x3FFFFu) >> 4) | (1u << 16); }

// D(tmem) (+)= A * B^T with both operands in shared memory, given the low
// descriptor words.
__device__ __forceinline__ void tc_mma_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " .reg .b64 da, db;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " mov.b64 da, {%1, %5};\n"
      " mov.b64 db, {%2, %5};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi)
      : "memory");
}

// D(tmem) (+)= A(tmem) * B^T, B in shared memory given its low descriptor word.
__device__ __forceinline__ void tc_mma_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " .reg .b64 db;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " mov.b64 db, {%2, %5};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi)
      : "memory");
}

// Eight MMAs over one 128-deep K extent of K-major operands in the 128-byte
// swizzle (two blocks of 64 columns, 16 KB apart for 128 rows): operand k
// starts 32 bytes (low-word step 2) after operand k-1 within a block and
// 1024 low-word units later in the second block.  The first MMA accumulates
// if `acc` is non-zero, the other seven always.  One asm statement, so the
// issuing warp spends no instructions re-deriving the predicate and the
// 64-bit descriptors between the MMAs.  Called by a whole converged warp
// with warp-uniform operands: one lane, chosen by elect.sync, issues; the
// descriptor arithmetic stays warp-uniform, which measured 7 % faster in
// the attention kernel than issuing from a single-lane branch.
__device__ __forceinline__ void tc_mma_ss_k128(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                               uint32_t acc) {
  asm volatile(
      "{\n"
      " .reg .pred p, t, e;\n"
      " elect.sync _|e, 0xffffffff;\n"
      " .reg .b64 da, db;\n"
      " .reg .b32 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " setp.eq.b32 t, %4, %4;\n"
      " mov.b64 da, {%1, %5};\n"
      " mov.b64 db, {%2, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n"
      " add.u32 a, %1, 2;\n"
      " add.u32 b, %2, 2;\n"
      " mov.b64 da, {a, %5};\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
      " add.u32 a, %1, 4;\n"
      " add.u32 b, %2, 4;\n"
      " mov.b64 da, {a, %5};\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
      " add.u32 a, %1, 6;\n"
      " add.u32 b, %2, 6;\n"
      " mov.b64 da, {a, %5};\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
      " add.u32 a, %1, 1024;\n"
      " add.u32 b, %2, 1024;\n"
      " mov.b64 da, {a, %5};\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
      " add.u32 a, %1, 1026;\n"
      " add.u32 b, %2, 1026;\n"
      " mov.b64 da, {a, %5};\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
      " add.u32 a, %1, 1028;\n"
      " add.u32 b, %2, 1028;\n"
      " mov.b64 da, {a, %5};\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
      " add.u32 a, %1, 1030;\n"
      " add.u32 b, %2, 1030;\n"
      " mov.b64 da, {a, %5};\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(acc), "r"(kDescHi)
      : "memory");
}
// The same with A read from tensor memory: operand k is 8 columns (16 BF16
// keys as pairs) after operand k-1.
__device__ __forceinline__ void tc_mma_ts_k128(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                               uint32_t acc) {
  asm volatile(
      "{\n"
      " .reg .pred p, t, e;\n"
      " elect.sync _|e, 0xffffffff;\n"
      " .reg .b64 db;\n"
      " .reg .b32 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " setp.eq.b32 t, %4, %4;\n"
      " mov.b64 db, {%2, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n"
      " add.u32 a, %1, 8;\n"
      " add.u32 b, %2, 2;\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %3, t;\n"
      " add.u32 a, %1, 16;\n"
      " add.u32 b, %2, 4;\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %3, t;\n"
      " add.u32 a, %1, 24;\n"
      " add.u32 b, %2, 6;\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %3, t;\n"
      " add.u32 a, %1, 32;\n"
      " add.u32 b, %2, 1024;\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %3, t;\n"
      " add.u32 a, %1, 40;\n"
      " add.u32 b, %2, 1026;\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %3, t;\n"
      " add.u32 a, %1, 48;\n"
      " add.u32 b, %2, 1028;\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %3, t;\n"
      " add.u32 a, %1, 56;\n"
      " add.u32 b, %2, 1030;\n"
      " mov.b64 db, {b, %5};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %3, t;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(acc), "r"(kDescHi)
      : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per
// thread), loaded and waited for in one statement so no use of the
// registers can be scheduled ahead of the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes, loaded and
// waited for in one statement.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 128 consecutive fp32 columns of this warp's 32 TMEM lanes in one load,
// waited for in the same statement.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 32 fp32 columns back to this warp's 32 TMEM lanes and wait.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
      " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Store 32 32-bit columns (e.g. packed BF16 pairs) to this warp's 32 TMEM
// lanes and wait.
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
      " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// ----------------------------------------------------------------- CTA pairs (cta_group::2)
// A pair of CTAs (ranks 0 and 1 of a cluster of 2) shares one tensor-core
// operation: rank 0 issues tcgen05.mma.cta_group::2 with M = 256, whose A
// rows 0..127 and B rows (N) 0..N/2-1 come from rank 0's shared memory and
// A rows 128..255 and B rows N/2..N-1 from rank 1's, at the same offsets;
// each CTA's tensor memory receives its own 128 rows.  The tensor memory of
// both is allocated and freed by one warp of each CTA together, and every
// tcgen05 instruction of such a kernel uses cta_group::2.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive once on the mbarrier at offset `bar` in every CTA of `mask` when
// all tcgen05 operations this thread issued so far have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// D (+)= A * B^T over the pair, both operands in shared memory, given the
// low descriptor words (the same offsets in both CTAs).
__device__ __forceinline__ void tc_mma_pair_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " .reg .b64 da, db;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " mov.b64 da, {%1, %5};\n"
      " mov.b64 db, {%2, %5};\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi)
      : "memory");
}
// TMA tile load into this CTA's shared memory whose completion is counted
// on an mbarrier that may sit in the peer CTA (bar: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
// Four MMAs over one 64-deep K block (K16 steps 32 bytes apart: low-word
// step 2 for both operands), cta_group::1 or ::2, issued by the elected lane
// of a whole converged warp (see tc_mma_ss_k128).  The first accumulates if
// `acc` is non-zero, the other three always.
template <bool PAIR>
__device__ __forceinline__ void tc_mma_k64_elect(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                                 uint32_t acc) {
  if constexpr (PAIR) {
    asm volatile(
        "{\n"
        " .reg .pred p, t, e;\n"
        " .reg .b64 da, db;\n"
        " .reg .b32 a, b;\n"
        " elect.sync _|e, 0xffffffff;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " setp.eq.b32 t, %4, %4;\n"
        " mov.b64 da, {%1, %5};\n mov.b64 db, {%2, %5};\n"
        " @e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, p;\n"
        " add.u32 a, %1, 2;\n add.u32 b, %2, 2;\n mov.b64 da, {a, %5};\n mov.b64 db, {b, %5};\n"
        " @e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, t;\n"
        " add.u32 a, %1, 4;\n add.u32 b, %2, 4;\n mov.b64 da, {a, %5};\n mov.b64 db, {b, %5};\n"
        " @e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, t;\n"
        " add.u32 a, %1, 6;\n add.u32 b, %2, 6;\n mov.b64 da, {a, %5};\n mov.b64 db, {b, %5};\n"
        " @e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, t;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(acc), "r"(kDescHi)
        : "memory");
  } else {
    asm volatile(
        "{\n"
        " .reg .pred p, t, e;\n"
        " .reg .b64 da, db;\n"
        " .reg .b32 a, b;\n"
        " elect.sync _|e, 0xffffffff;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " setp.eq.b32 t, %4, %4;\n"
        " mov.b64 da, {%1, %5};\n mov.b64 db, {%2, %5};\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n"
        " add.u32 a, %1, 2;\n add.u32 b, %2, 2;\n mov.b64 da, {a, %5};\n mov.b64 db, {b, %5};\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
        " add.u32 a, %1, 4;\n add.u32 b, %2, 4;\n mov.b64 da, {a, %5};\n mov.b64 db, {b, %5};\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
        " add.u32 a, %1, 6;\n add.u32 b, %2, 6;\n mov.b64 da, {a, %5};\n mov.b64 db, {b, %5};\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(acc), "r"(kDescHi)
        : "memory");
  }
}
// tcgen05.commit over the pair (multicast to the CTAs of `mask`) from a
// whole converged warp: one elected lane commits.
__device__ __forceinline__ void tc_commit_pair_elect(uint32_t bar, uint16_t mask) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}\n"
      ::"r"(bar), "h"(mask)
      : "memory");
}
// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address),
// with the default (CTA-scope) release: the tensor-memory accesses it
// orders are covered by tcgen05.fence::before_thread_sync on this side and
// ::after_thread_sync on the waiting side, and a cluster-scope release
// measured 1000-1700 cycles per arrive.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// ----------------------------------------------------------------- packing
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

// Packed fp32 pairs on the FMA pipe (sm_100 family): one instruction for
// two lanes' worth of arithmetic.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
  asm("{\n"
      " .reg .b64 ra, rb, rc, rd;\n"
      " mov.b64 ra, {%2, %3};\n"
      " mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n"
      " mov.b64 {%0, %1}, rd;\n"
      "}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n"
      " .reg .b64 ra, rb, rd;\n"
      " mov.b64 ra, {%2, %3};\n"
      " mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;\n"
      "}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// max of three (sm_100 family)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace h3
