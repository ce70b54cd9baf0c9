// tcgen05 / TMA / mbarrier wrappers shared by the tensor-core GEMM kernels
// (inline PTX for sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "sq_async.cuh"

namespace sq {
namespace tc {
using async::su32;

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

SQ_DEVINL void mbar_init(uint64_t* b, uint32_t count) { async::mbar_init(b, count); }
SQ_DEVINL void mbar_expect_tx(uint64_t* b, uint32_t bytes) { async::mbar_expect_tx(b, bytes); }
SQ_DEVINL bool mbar_try_wait(uint64_t* b, uint32_t parity) { return async::mbar_try_wait(b, parity); }
SQ_DEVINL uint64_t global_ns() { return async::global_ns(); }

// Arrive on an mbarrier given by its shared::cluster address (this CTA's
// or the peer's).  The barriers this is used on order tensor-memory reads
// (completed by tcgen05.wait::ld, fenced by tcgen05.fence around the
// arrive/wait pair) before the MMAs that overwrite the same columns; no
// generic-memory data passes through them, so the default CTA-scope release
// is enough (a cluster-scope release costs a memory barrier per arrive).
SQ_DEVINL void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// Arrive with release at cluster scope on an mbarrier given by its
// shared::cluster address: orders this thread's earlier memory operations
// (and, after fence.proxy.async, its shared-memory writes as the tensor
// cores see them) before the phase completion that a waiter in either CTA
// of the cluster acquires.
SQ_DEVINL void mbar_arrive_release_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// try_wait with acquire at cluster scope, for phases completed by arrivals
// from the peer CTA.
SQ_DEVINL bool mbar_try_wait_acq_cluster(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait at cluster scope without ordering (relaxed); a successful poll is
// followed by fence_acq_rel_cluster, which gives it acquire semantics at
// cluster scope once instead of on every poll.
SQ_DEVINL bool mbar_try_wait_relaxed_cluster(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
SQ_DEVINL void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (tensor-core operand reads, TMA).
SQ_DEVINL void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Bounded wait for the phase with parity `parity` to complete.  Returns
// false if the CTA is aborting or the wait ran out (which starts the abort).
// With CLUSTER_ACQ the wait acquires at cluster scope: relaxed polls at
// cluster scope, then one cluster-scope fence once the phase has completed.
template <bool CLUSTER_ACQ = false>
SQ_DEVINL bool mbar_wait(uint64_t* b, uint32_t parity, int* abort_flag, int32_t* flags,
                         uint64_t limit_ns = WAIT_LIMIT_NS) {
  auto poll = [&] {
    if (!CLUSTER_ACQ) return mbar_try_wait(b, parity);
    if (!mbar_try_wait_relaxed_cluster(b, parity)) return false;
    fence_acq_rel_cluster();
    return true;
  };
  if (poll()) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (poll()) return true;
    if ((i & 63) == 0) {
      if (*(volatile int*)abort_flag) return false;
      if (global_ns() - t0 > limit_ns) {
        *(volatile int*)abort_flag = 1;
        raise_flag(flags, SQ_FLAG_TIMEOUT);
        return false;
      }
    }
  }
}

// TMA load of box (x, y) into this CTA's shared memory, completing on the
// mbarrier at shared::cluster address `bar` (with CG = 2, the even CTA's
// barrier, which counts both CTAs' bytes).
template <int CG>
SQ_DEVINL void tma_load(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  if constexpr (CG == 2) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
        "[%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
  }
}

SQ_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SQ_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major tile stored as 128-byte rows
// with the 128-byte swizzle (what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B):
// start address >> 4 in bits 0-13, leading byte offset (unused by this
// layout) 16 >> 4 in bits 16-29, stride byte offset between 8-row groups
// 1024 >> 4 in bits 32-45, the fixed value 1 in bits 46-48, base offset 0,
// and swizzle mode 2 (128 B) in bits 61-63.
SQ_DEVINL uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

template <int CG>
SQ_DEVINL void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                        uint32_t accumulate) {
  if constexpr (CG == 2) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Arrive (once) on `bar` when every MMA this thread issued so far has
// completed; with CG = 2 on the barrier at the same offset in both CTAs.
template <int CG>
SQ_DEVINL void mma_commit(uint64_t* bar) {
  if constexpr (CG == 2) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(su32(bar)),
        "h"(mask)
        : "memory");
  } else {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     su32(bar))
                 : "memory");
  }
}

template <int CG, uint32_t TMEM_COLS>
SQ_DEVINL void tmem_alloc(uint32_t* dst) {
  if constexpr (CG == 2) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(dst)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(dst)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
}

template <int CG, uint32_t TMEM_COLS>
SQ_DEVINL void tmem_dealloc(uint32_t taddr) {
  if constexpr (CG == 2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(TMEM_COLS)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(TMEM_COLS)
                 : "memory");
}

// 8 consecutive fp32 accumulator columns of this warp's 32 lanes.
SQ_DEVINL void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
}
SQ_DEVINL void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

SQ_DEVINL int32_t f32_to_i32_exact(uint32_t bits) {
  int32_t v;
  asm("cvt.rni.s32.f32 %0, %1;" : "=r"(v) : "f"(__uint_as_float(bits)));
  return v;
}

}  // namespace tc
}  // namespace sq
