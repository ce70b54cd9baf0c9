// mbarrier, bulk-copy (TMA) and cluster primitives shared by the streaming
// kernels of the sm_103a library, written as inline PTX.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "sq_common.cuh"

namespace sq {
namespace async {

SQ_DEVINL uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

SQ_DEVINL void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the async proxy (TMA) and, with a
// cluster, to the other CTAs of the cluster.
SQ_DEVINL void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

SQ_DEVINL void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}

SQ_DEVINL void mbar_arrive_local(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

SQ_DEVINL bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, "
      "p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

SQ_DEVINL uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `parity` to complete, for at most limit_ns
// nanoseconds.  Returns false if the wait ran out.
SQ_DEVINL bool mbar_wait_bounded(uint64_t* b, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 31) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}

// One-dimensional bulk copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on mbarrier `bar`.  Both addresses 16-byte
// aligned, bytes a multiple of 16.
SQ_DEVINL void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (the policy from createpolicy).
SQ_DEVINL void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar)), "l"(policy)
      : "memory");
}

SQ_DEVINL uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Two-dimensional tiled TMA load of box (x, y) of `map` into shared memory.
SQ_DEVINL void tma_load_2d(void* dst, const void* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}

SQ_DEVINL void prefetch_tensormap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Two-dimensional tiled TMA store of the box at (x, y) of `map` from shared
// memory, tracked by this thread's bulk groups.  The box's part outside the
// tensor is not written.
SQ_DEVINL void tma_store_2d(const void* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(su32(src)), "r"(x), "r"(y)
               : "memory");
}
SQ_DEVINL void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's committed bulk stores have finished reading shared memory
SQ_DEVINL void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's committed bulk stores are complete
SQ_DEVINL void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy writes to shared memory become visible to the async proxy
SQ_DEVINL void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------------------ clusters
SQ_DEVINL uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

SQ_DEVINL void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
SQ_DEVINL void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Shared-memory address of the same variable in CTA `rank` of the cluster.
SQ_DEVINL uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

SQ_DEVINL uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// ------------------------------------------------------------------ packed fp32
// Two IEEE binary32 operations per instruction, each rounded to nearest
// even like its scalar form.  Use them only where no add consumes a
// multiply's result: a packed multiply followed by a packed add was seen to
// round like a fused multiply-add (a tie of the product rounded the other
// way), so the quantizers do that pair in scalar mul.rn/add.rn, which are
// never contracted.
SQ_DEVINL void mul2_rn(float& a0, float& a1, float b0, float b1) {
  asm("{\n.reg .b64 x, y;\nmov.b64 x, {%0, %1};\nmov.b64 y, {%2, %3};\nmul.rn.f32x2 x, x, y;\n"
      "mov.b64 {%0, %1}, x;\n}\n"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}
SQ_DEVINL void add2_rn(float& a0, float& a1, float b0, float b1) {
  asm("{\n.reg .b64 x, y;\nmov.b64 x, {%0, %1};\nmov.b64 y, {%2, %3};\nadd.rn.f32x2 x, x, y;\n"
      "mov.b64 {%0, %1}, x;\n}\n"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

SQ_DEVINL void fma2_rn(float& a0, float& a1, float b0, float b1, float c0, float c1) {
  // (a0, a1) = (RN(a0 * b0 + c0), RN(a1 * b1 + c1)), each one fused multiply-add
  asm("{\n.reg .b64 x, y, z;\nmov.b64 x, {%0, %1};\nmov.b64 y, {%2, %3};\nmov.b64 z, {%4, %5};\n"
      "fma.rn.f32x2 x, x, y, z;\nmov.b64 {%0, %1}, x;\n}\n"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Two quotients RN(v0 / d0), RN(v1 / d1) by quot_rn's sequence (sq_common.cuh:
// y = RN(1/d), one multiply and four fused multiply-adds, Markstein's
// correction), two lanes per instruction; the same preconditions.
SQ_DEVINL void quot2_rn(float& v0, float& v1, float d0, float d1, float y0, float y1) {
  float q0 = v0, q1 = v1;
  mul2_rn(q0, q1, y0, y1);
  float r0 = -d0, r1 = -d1;
  fma2_rn(r0, r1, q0, q1, v0, v1);   // v - d q
  fma2_rn(r0, r1, y0, y1, q0, q1);   // q + r y
  q0 = r0;
  q1 = r1;
  r0 = -d0;
  r1 = -d1;
  fma2_rn(r0, r1, q0, q1, v0, v1);
  fma2_rn(r0, r1, y0, y1, q0, q1);
  v0 = r0;
  v1 = r1;
}

// max(|m|, |v|) in magnitude, NaN if either is NaN; the sign of the result
// is meaningless (callers take the magnitude at the end).
SQ_DEVINL float absmax_nan(float m, float v) {
  float r;
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(v));
  return r;
}

// The same on two packed bfloat16 values per word (exact: a maximum of
// magnitudes needs no rounding).
SQ_DEVINL uint32_t absmax_nan_bf16x2(uint32_t m, uint32_t v) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(v));
  return r;
}

// ------------------------------------------------------------------ host side
// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

}  // namespace async
}  // namespace sq
