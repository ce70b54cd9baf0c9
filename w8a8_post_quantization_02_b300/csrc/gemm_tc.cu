// Step 5, tensor-core path: INT8 x INT8 GEMM on sm_103a's tcgen05 tensor
// cores, with exact integer accumulation and the bf16 dequantizing epilogue.
//
// Source: learn-kernels.com "Quantization", paragraph 2: both operands of
// the matmul are INT8 and the product runs on the low-precision hardware
// path; paragraph 1: prefill is compute-bound.
//
// sm_103a's tcgen05.mma has no integer kind, so the INT8 codes arrive as
// exact bfloat16 values (|code| <= 127 needs 7 significand bits) and the
// MMA runs as kind::f16 with fp32 accumulation in tensor memory.  Every
// product is an integer of magnitude <= 127^2 and every partial sum of at
// most 1024 products stays below 2^24, so the fp32 accumulator holds it
// exactly.  The K loop is therefore cut into chunks of 1024: after each
// chunk the epilogue warps read the fp32 accumulator from TMEM, convert it
// to int32 (exact) and add it to int32 running sums held in registers; the
// MMA warp meanwhile fills the other of two TMEM accumulator buffers.
//
// Kernel shape: persistent, one CTA per SM, 128 x 256 output tiles,
// 4-stage TMA pipeline of 128 x 64 (A) and 256 x 64 (B) bf16 tiles in
// 128-byte-swizzled shared memory.  Warp 0 issues TMA loads, warp 1 owns
// TMEM and issues the MMAs, warps 2-9 drain the accumulators and write Y.
// Every mbarrier wait is bounded in time; a wait that runs out sets
// SQ_FLAG_TIMEOUT, stops the CTA's loops, waits for its own outstanding
// copies and MMAs (also bounded), frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "sq_common.cuh"

namespace sq {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int CHUNK_KB = 16;  // k-blocks of 64 per exact fp32 chunk (1024 products)
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = (2 + EPI_WARPS) * 32;
constexpr uint32_t TMEM_COLS = 2 * BN;  // two fp32 accumulator buffers
constexpr int COLS_PER_EPI_WARP = BN / 2;
// instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

struct Smem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;  // + alignment slack

// ------------------------------------------------------------------ PTX wrappers
SQ_DEVINL uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

SQ_DEVINL void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
SQ_DEVINL void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}
SQ_DEVINL void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
SQ_DEVINL bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
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
// Bounded wait for the phase with parity `parity` to complete.  Returns
// false if the CTA is aborting or the wait ran out (which starts the abort).
SQ_DEVINL bool mbar_wait(uint64_t* b, uint32_t parity, Smem& sm, int32_t* flags,
                         uint64_t limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 0) {
      if (*(volatile int*)&sm.abort) return false;
      if (global_ns() - t0 > limit_ns) {
        *(volatile int*)&sm.abort = 1;
        raise_flag(flags, SQ_FLAG_TIMEOUT);
        return false;
      }
    }
  }
}

SQ_DEVINL void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
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

SQ_DEVINL void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
      : "memory");
}
SQ_DEVINL void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   su32(bar))
               : "memory");
}

#define SQ_R32(i) "=r"(r[i])
SQ_DEVINL void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : SQ_R32(0), SQ_R32(1), SQ_R32(2), SQ_R32(3), SQ_R32(4), SQ_R32(5), SQ_R32(6), SQ_R32(7),
        SQ_R32(8), SQ_R32(9), SQ_R32(10), SQ_R32(11), SQ_R32(12), SQ_R32(13), SQ_R32(14), SQ_R32(15),
        SQ_R32(16), SQ_R32(17), SQ_R32(18), SQ_R32(19), SQ_R32(20), SQ_R32(21), SQ_R32(22),
        SQ_R32(23), SQ_R32(24), SQ_R32(25), SQ_R32(26), SQ_R32(27), SQ_R32(28), SQ_R32(29),
        SQ_R32(30), SQ_R32(31)
      : "r"(taddr));
}
#undef SQ_R32
SQ_DEVINL void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

SQ_DEVINL int32_t f32_to_i32_exact(uint32_t bits) {
  int32_t v;
  asm("cvt.rni.s32.f32 %0, %1;" : "=r"(v) : "f"(__uint_as_float(bits)));
  return v;
}

struct Problem {
  int64_t M, N, K;
  int tiles_m, tiles_n, n_kb, n_chunks;
  int vec_ok;  // N % 8 == 0 and y / acc_out 16-byte aligned: 16-byte stores
};

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_bf16c(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const float* __restrict__ x_scale, const float* __restrict__ w_scale,
                 __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out, int32_t* flags,
                 Problem P) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = P.tiles_m * P.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], EPI_WARPS);
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&sm.tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m0 = (tile % P.tiles_m) * BM, n0 = (tile / P.tiles_m) * BN;
        for (int kb = 0; kb < P.n_kb; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1, sm, flags)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.full[stage], STAGE_BYTES);
          tma_load_2d(sm.a[stage], &map_a, &sm.full[stage], kb * BK, m0);
          tma_load_2d(sm.b[stage], &map_b, &sm.full[stage], kb * BK, n0);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA exits
        for (int i = 0; i < STAGES && issued > 0; ++i, --issued) {
          if (--stage < 0) {
            stage = STAGES - 1;
            phase ^= 1;
          }
          uint64_t t0 = global_ns();
          while (!mbar_try_wait(&sm.full[stage], phase) && global_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t chunk_ctr = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        for (int c = 0; ok && c < P.n_chunks; ++c) {
          const uint32_t buf = chunk_ctr & 1, use = chunk_ctr >> 1;
          if (!mbar_wait(&sm.acc_empty[buf], (use & 1) ^ 1, sm, flags)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + buf * BN;
          const int kb0 = c * CHUNK_KB, kb1 = min(P.n_kb, kb0 + CHUNK_KB);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&sm.full[stage], phase, sm, flags)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = su32(sm.a[stage]), b_addr = su32(sm.b[stage]);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_bf16(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32),
                       (kb > kb0 || kk > 0) ? 1u : 0u);
            mma_commit(&sm.empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          mma_commit(&sm.acc_full[buf]);
          ++chunk_ctr;
        }
      }
      // wait for every MMA this thread issued before TMEM is released
      mma_commit(&sm.drain);
      uint64_t t0 = global_ns();
      while (!mbar_try_wait(&sm.drain, 0) && global_ns() - t0 < WAIT_LIMIT_NS) {
      }
    }
  } else {
    // ---------------- epilogue warps: drain chunks, then write Y
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;       // which 128 columns of the 256
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t chunk_ctr = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const int64_t m0 = (int64_t)(tile % P.tiles_m) * BM, n0 = (int64_t)(tile / P.tiles_m) * BN;
      int32_t acc[COLS_PER_EPI_WARP];
#pragma unroll
      for (int i = 0; i < COLS_PER_EPI_WARP; ++i) acc[i] = 0;
      for (int c = 0; c < P.n_chunks; ++c) {
        const uint32_t buf = chunk_ctr & 1, use = chunk_ctr >> 1;
        // one lane waits and the warp follows its verdict, so the warp stays
        // converged for the .sync.aligned TMEM loads
        int got = 1;
        if (lane == 0) got = mbar_wait(&sm.acc_full[buf], use & 1, sm, flags) ? 1 : 0;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
        const uint32_t base = tmem + lane_base + buf * BN + half * COLS_PER_EPI_WARP;
#pragma unroll
        for (int j = 0; j < COLS_PER_EPI_WARP / 64; ++j) {
          uint32_t r0[32], r1[32];
          tmem_ld32(base + j * 64, r0);
          tmem_ld32(base + j * 64 + 32, r1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            acc[j * 64 + i] += f32_to_i32_exact(r0[i]);
            acc[j * 64 + 32 + i] += f32_to_i32_exact(r1[i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
        ++chunk_ctr;
      }
      if (!ok) break;
      const int64_t m = m0 + q * 32 + lane;
      if (m < P.M) {
        const float xs = x_scale[m];
        const int64_t nb = n0 + half * COLS_PER_EPI_WARP;
#pragma unroll
        for (int g = 0; g < COLS_PER_EPI_WARP / 8; ++g) {
          const int64_t n = nb + g * 8;
          if (n >= P.N) break;
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float ws = (n + e < P.N) ? __ldg(w_scale + n + e) : 0.0f;
            v[e] = __fmul_rn(__fmul_rn(__int2float_rn(acc[g * 8 + e]), xs), ws);
          }
          __nv_bfloat16* yrow = y + m * P.N + n;
          if (n + 8 <= P.N && P.vec_ok) {
            uint4 o;
            o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[0])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[1])) << 16);
            o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[3])) << 16);
            o.z = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[4])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[5])) << 16);
            o.w = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[6])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[7])) << 16);
            st16(yrow, o);
            if (acc_out) {
              int32_t* arow = acc_out + m * P.N + n;
              st16(arow, make_uint4(acc[g * 8 + 0], acc[g * 8 + 1], acc[g * 8 + 2], acc[g * 8 + 3]));
              st16(arow + 4, make_uint4(acc[g * 8 + 4], acc[g * 8 + 5], acc[g * 8 + 6], acc[g * 8 + 7]));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (n + e < P.N) {
                yrow[e] = __float2bfloat16_rn(v[e]);
                if (acc_out) acc_out[m * P.N + n + e] = acc[g * 8 + e];
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows x k] (k contiguous), box of 64 x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)k * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tc

sq_status gemm_bf16c_tc(const void* xq, const float* x_scale, const void* wq, const float* w_scale,
                        int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                        cudaStream_t st) {
  using namespace tc;
  if (m > (int64_t)1 << 31 || n > (int64_t)1 << 31 || k > (int64_t)1 << 31) return SQ_ERR_UNSUPPORTED;
  CUtensorMap ma, mb;
  if (!make_map(&ma, xq, m, k, BM) || !make_map(&mb, wq, n, k, BN)) return SQ_ERR_CUDA;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_gemm_bf16c, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
      return SQ_ERR_CUDA;
    attr_set = true;
  }
  Problem P;
  P.M = m;
  P.N = n;
  P.K = k;
  P.tiles_m = (int)((m + BM - 1) / BM);
  P.tiles_n = (int)((n + BN - 1) / BN);
  P.n_kb = (int)((k + BK - 1) / BK);
  P.n_chunks = (P.n_kb + CHUNK_KB - 1) / CHUNK_KB;
  P.vec_ok = (n % 8 == 0) && aligned16(y) && (acc_out == nullptr || aligned16(acc_out));
  const int tiles = P.tiles_m * P.tiles_n;
  const int grid = std::min(tiles, sm_count());
  k_gemm_bf16c<<<grid, THREADS, SMEM_BYTES, st>>>(ma, mb, x_scale, w_scale,
                                                   static_cast<__nv_bfloat16*>(y), acc_out, flags, P);
  return launch_status();
}

}  // namespace sq
