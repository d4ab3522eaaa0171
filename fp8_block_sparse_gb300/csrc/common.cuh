// common.cuh -- sm_103a building blocks shared by the kernels of libmsa.so:
// bounded mbarrier waits, TMA tensor loads, tcgen05 (TMEM allocation, MMA,
// commit, TMEM loads/stores) and the shared-memory / instruction descriptors.
//
// Every wait on an mbarrier is bounded by wall-clock time (globaltimer). A
// wait that runs out records MSA_DEVERR_TIMEOUT in the device error word and
// returns false; callers then stop issuing work and leave cleanly. Nothing
// here traps.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace msa {

// Wall-clock limit of one bounded wait (ns). No wait in these kernels is
// legitimately longer than a few milliseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

#define MSA_DEV __device__ __forceinline__

MSA_DEV uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MSA_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- dependent launch
// pdl_wait: blocks until the kernel this one follows in the stream has
// completed and its writes are visible (a no-op when it was launched
// without programmatic serialisation). Nothing may read what the previous
// kernel writes, or write what it reads, before this point.
MSA_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// pdl_trigger: lets the next kernel's blocks be scheduled once every block
// of this one has triggered or exited. Kernels that allocate tensor memory
// trigger only after their allocation, so a waiting dependent block never
// holds columns that a block of this kernel still needs to allocate.
MSA_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
MSA_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
MSA_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MSA_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
MSA_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
MSA_DEV uint32_t mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok;
}
// Waits for the phase with the given parity to complete. Returns false (and
// records a timeout) when the wall-clock limit runs out first.
MSA_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, MSA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Values of a CTA's shared abort flag: 0 = run; 1 = some wait of this CTA
// ran out, every role stops waiting; kAbortForced = the device's debug switch
// that forces timeouts is on: the first wait that is not complete at its
// first test gives up at once (then the flag becomes 1).
constexpr int kAbortForced = 2;

// The initial value of a CTA's abort flag (read once, at kernel start, from
// the per-device state that `err` points into).
MSA_DEV int initial_abort(const unsigned* err) {
  return reinterpret_cast<const volatile DeviceState*>(err)->force_timeouts ? kAbortForced : 0;
}

// As mbar_wait, but returns false at once when *abort is set, and sets it
// when its own limit runs out: after the first timeout every role of the CTA
// stops waiting and drains its loop quickly.
MSA_DEV bool mbar_wait_ab(uint64_t* bar, uint32_t parity, unsigned* err, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    const int ab = *abort;
    if (ab) {
      if (ab == kAbortForced) {
        atomicOr(err, MSA_DEVERR_TIMEOUT);
        *abort = 1;
      }
      return false;
    }
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, MSA_DEVERR_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// Exit-path drain of a ring of `stages` barriers whose iterations 0..n-1 were
// each armed with an asynchronous copy (or completed by an arrival): waits,
// with the fixed limit and regardless of the abort flag, for the last armed
// phase of every stage. Phases of one barrier complete in order, so after
// this no copy issued into the ring is still writing shared memory.
MSA_DEV void mbar_drain_ring(uint64_t* bars, int stages, int n, unsigned* err) {
  for (int s = 0; s < stages && s < n; ++s) {
    const int j = s + ((n - 1 - s) / stages) * stages;       // last iteration on stage s
    mbar_wait(&bars[s], uint32_t((j / stages) & 1), err);
  }
}

// ---------------------------------------------------------------- TMA
MSA_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
MSA_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}
MSA_DEV void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Tiled TMA store of one box from shared memory (bulk-group completion):
// bulk_commit() closes the group, bulk_wait_read() waits until the copies
// have read their shared-memory source (it may then be reused or released).
MSA_DEV void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(src)), "r"(x), "r"(y)
      : "memory");
}
MSA_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
MSA_DEV void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Plain bulk copy global -> shared (both 16-byte aligned, size a multiple of 16).
MSA_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// 16-byte asynchronous global -> shared copy (L2 only); writes 16 zero
// bytes instead (no global read) when !valid.
MSA_DEV void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16u : 0u)
               : "memory");
}
// Arrives on `bar` once every cp.async this thread issued so far has
// landed; the barrier's count must include these arrivals (no increment).
MSA_DEV void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
MSA_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.mma operands written by threads).
MSA_DEV void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05
// TMEM allocation is a warp-wide operation; the base address is written to smem.
MSA_DEV void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
MSA_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MSA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MSA_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MSA_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Instruction descriptor: dense, fp32 accumulator, A/B format code 0 (E4M3 for
// kind::f8f6f4, F16 for kind::f16), both operands K-major (callers OR in bit
// 15 / 16 for an MN-major A / B), no negation.
__host__ __device__ constexpr uint32_t idesc_f32(int M, int N) {
  return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major operand in the canonical
// swizzled layout: rows of `swz` bytes (128 or 64), 8-row groups of 8*swz
// bytes stacked along M/N, the 16-byte chunks of row r XOR-ed with (r % 8).
// The region must be aligned to 8*swz bytes; a K offset inside the swizzle
// row is applied by adding its byte offset to saddr.
MSA_DEV uint64_t sdesc_kmajor(uint32_t saddr, uint32_t swz) {
  const uint64_t layout = (swz == 128) ? 2ull : (swz == 64 ? 4ull : 6ull);
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t(1) << 16) |
         (uint64_t(((8u * swz) >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (layout << 61);
}

// Shared-memory matrix descriptor for an MN-major operand in the 128-byte
// swizzled layout: rows of 128 bytes along M/N (64 f16 or 128 e4m3), one row
// per K index, 8-row groups 1024 bytes apart along K, and successive 128-byte
// wide column blocks of M/N `mn_stride` bytes apart. Select it with the
// transpose bit of the instruction descriptor (bit 15 for A, 16 for B).
MSA_DEV uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t mn_stride) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((mn_stride >> 4) & 0x3FFFu) << 16) |
         (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Byte offset of the 16-byte chunk `c` of row `r` inside a swizzled K-major
// region with `swz`-byte rows (the layout TMA writes with the same swizzle):
// address bits [4, 4+n) are XOR-ed with bits [7, 7+n), n = log2(swz/16).
MSA_DEV uint32_t swz_offset(uint32_t r, uint32_t c, uint32_t swz) {
  const uint32_t o = r * swz + c * 16u;
  return o ^ (((o >> 7) & (swz / 16u - 1u)) << 4);
}

// TMEM address: lane in bits 31..16, column in bits 15..0.
MSA_DEV uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32*(w%4) .. +31). Load and wait are fused so the values are ready on return.
MSA_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 64 consecutive fp32 columns of this thread's TMEM lane, load + wait fused.
MSA_DEV void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}
// Store of 16 columns without waiting; tmem_wait_st2 then waits for every
// store this thread issued, taking the two 16-register sources as in-out
// operands so neither is reused before the stores have read it.
MSA_DEV void tmem_st16_async(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
MSA_DEV void tmem_wait_st2(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.wait::st.sync.aligned;"
      : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
        "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]),
        "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
        "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15])
      :
      : "memory");
}
// 16 consecutive fp32 columns, load + wait fused.
MSA_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// 8 / 4 consecutive 32-bit columns of this thread's TMEM lane, load + wait fused.
MSA_DEV void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
}
MSA_DEV void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(taddr)
      : "memory");
}
// Store 8 / 4 consecutive 32-bit columns to this thread's TMEM lane, then wait.
MSA_DEV void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
MSA_DEV void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
      : "memory");
}
// Column loads/stores of a compile-time width 4 or 8.
template <int N>
MSA_DEV void tmem_ldn(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 8) tmem_ld8(taddr, r); else tmem_ld4(taddr, r);
}
template <int N>
MSA_DEV void tmem_stn(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 8) tmem_st8(taddr, r); else tmem_st4(taddr, r);
}
// Store 32 consecutive 32-bit columns to this thread's TMEM lane, then wait.
MSA_DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Store 16 fp32 columns to this thread's TMEM lane, store + wait fused.
MSA_DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// ---------------------------------------------------------------- warp-issued tcgen05
// tcgen05 MMAs (D[tmem] (+)= A * B^T, fp32 accumulate; A and B from shared
// memory descriptors, or A from TMEM for the _ts form) and commits, called by
// a whole converged warp with one lane elected inside the instruction
// sequence. Keeping the issuing loop converged lets the compiler hold
// descriptors and addresses in warp-uniform registers; a loop run by lane 0
// alone measurably slows every issue and turns each commit into a stall.
MSA_DEV void mma_e4m3_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// kind::f8f6f4 with the A operand (e4m3, four per 32-bit column, lane = row)
// in TMEM.
MSA_DEV void mma_e4m3_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
MSA_DEV void mma_f16_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
MSA_DEV void mma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_addr(bar))
      : "memory");
}
// Exit-path drain of the MMA-issuing warp (whole warp, converged): commits
// every tcgen05 operation it issued to `bar` (a barrier of count 1 used for
// nothing else) and waits for it with the fixed limit, regardless of the
// abort flag, so no MMA still reads shared memory or writes TMEM once the CTA
// frees them.
MSA_DEV void mma_drain_w(uint64_t* bar, unsigned* err);

// mbar_wait for a whole converged warp; the result is the same in every lane.
MSA_DEV bool mbar_wait_warp(uint64_t* bar, uint32_t parity, unsigned* err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err));
}
// mbar_wait_ab for a whole converged warp; the result is the same in every lane.
MSA_DEV bool mbar_wait_warp(uint64_t* bar, uint32_t parity, unsigned* err, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait_ab(bar, parity, err, abort));
}

MSA_DEV void mma_drain_w(uint64_t* bar, unsigned* err) {
  mma_commit_w(bar);
  mbar_wait_warp(bar, 0, err);
}

// ---------------------------------------------------------------- misc
// Two e4m3 codes (low byte first) -> two f16 (exact: every e4m3 value is an f16).
MSA_DEV uint32_t e4m3x2_to_f16x2(uint16_t x) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(x));
  return r;
}
// Two fp32 -> e4m3x2 (round to nearest even, saturating to +-448), `lo` in
// the low byte.
MSA_DEV uint16_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two fp32 -> f16x2 (round to nearest even), `lo` in the low half.
MSA_DEV uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two fp32 -> bf16x2 (round to nearest even), `lo` in the low half.
MSA_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Packed fp32 pairs (two lanes of one 64-bit register pair), sm_100+.
MSA_DEV uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
MSA_DEV float2 unpk2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
MSA_DEV uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
MSA_DEV uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
MSA_DEV float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

MSA_DEV uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
MSA_DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace msa
