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
// Kernel shape: persistent, 128 x 64 (A) and BN x 64 (B) bf16 tiles in
// 128-byte-swizzled shared memory fed by a TMA pipeline.  Warp 0 issues TMA
// loads, warp 1 owns TMEM and issues the MMAs, warps 2-9 drain the
// accumulators and write Y.
//   CG = 1: one CTA per SM computes 128 x BN output tiles.
//   CG = 2: a cluster of two CTAs on two SMs computes 256 x BN tiles with
//     tcgen05.mma.cta_group::2: each CTA loads its own 128 rows of A and
//     BN/2 rows of B, the even CTA issues M = 256 MMAs that read both CTAs'
//     shared memory and write each CTA's own 128 accumulator lanes.  Per
//     SM this moves 2/3 of the operand bytes of the one-CTA tile.
// BN (the output-channel tile, 256 or 240) is chosen per problem to fill
// the last wave of tiles.  With F16 the operands are exact fp16 values
// instead (the same integers; 1-byte codes widened by k_widen_codes below).  Every mbarrier wait is bounded in time; a wait that runs out
// sets SQ_FLAG_TIMEOUT, stops the CTA's loops, waits (bounded) for its own
// outstanding copies and MMAs, frees TMEM and returns.
#include "sq_tc.cuh"

#include <cstring>

namespace sq {
namespace tc {

constexpr int BM = 128;       // accumulator lanes (rows of A) per CTA
constexpr int BK = 64;        // 64 bf16 = one 128-byte swizzle row along K
constexpr int CHUNK_KB = 16;  // k-blocks of 64 per exact fp32 chunk (1024 products)
constexpr int A_BYTES = BM * BK * 2;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = (2 + EPI_WARPS) * 32;
constexpr uint32_t TMEM_COLS = 512;    // two accumulator buffers at columns 0 and 256
constexpr uint32_t TMEM_BUF_STRIDE = 256;

template <int CG, int BN>
struct Cfg {
  static constexpr int B_ROWS = BN / CG;                 // rows of B this CTA loads
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // this CTA's bytes per stage
  static constexpr int STAGES = (CG == 1 && BN > 128) ? 4 : 6;
  static constexpr int MMA_M = BM * CG;
  // instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
  // (bits 7-9 = 1, 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24
  // fp16 operands: A and B formats 0 in bits 7-9 and 10-12
  static constexpr uint32_t IDESC_F16 = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(MMA_M >> 4) << 24);
  static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                                    ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(MMA_M >> 4) << 24);
  static constexpr int COLS = BN / 2;  // accumulator columns per epilogue warp
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "MMA N");
  static_assert(B_ROWS % 8 == 0, "whole 8-row swizzle atoms");
  static_assert(COLS % 8 == 0, "epilogue works in 8-column groups");
  // Y leaves through shared memory: each epilogue warp stages 32 rows x
  // SLICE columns and stores them with one TMA copy.  40-column rows (80
  // bytes) are written without bank conflicts as they are; 32-column rows
  // (64 bytes) use the 64-byte swizzle.
  static constexpr int SLICE = COLS % 40 == 0 ? 40 : 32;
  static constexpr int SLICE_BYTES = 32 * SLICE * 2;
  static constexpr bool SW64 = SLICE == 32;
  static_assert(COLS % SLICE == 0 && SLICE % 8 == 0, "whole 16-byte groups per slice");
};

template <int CG, int BN>
struct Smem {
  using C = Cfg<CG, BN>;
  uint8_t a[C::STAGES][A_BYTES];
  uint8_t b[C::STAGES][C::B_BYTES];
  // each epilogue warp's w_scale slice for the current tile, loaded when the
  // tile starts so the output pass reads it from shared memory
  alignas(16) float ws[EPI_WARPS][C::COLS];
  alignas(1024) uint8_t ystage[EPI_WARPS][C::SLICE_BYTES];
  uint64_t full[C::STAGES];
  uint64_t empty[C::STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct Problem {
  int64_t M, N, K;
  int tiles_m, tiles_n, n_kb, n_chunks;
  int vec_ok;  // N % 8 == 0 and y / acc_out 16-byte aligned: 16-byte stores
  int tma_y;   // N % 8 == 0 and y 16-byte aligned: Y leaves by TMA stores
  int stall;   // the producer issues no copies (the bounded waits' test): 0 on every product call
  uint64_t wait_ns;  // bound on every pipeline wait
};

// Eight floats rounded to bf16, packed in column order.
SQ_DEVINL uint4 pack_bf16x8(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i])) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1])) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ------------------------------------------------------------------ kernel
template <int CG, int BN, bool F16>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_bf16c(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const __grid_constant__ CUtensorMap map_y,
                 const float* __restrict__ x_scale, const float* __restrict__ w_scale,
                 __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out, int32_t* flags,
                 Problem P) {
  using C = Cfg<CG, BN>;
  extern __shared__ uint8_t smem_raw[];
  Smem<CG, BN>& sm =
      *reinterpret_cast<Smem<CG, BN>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? async::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = blockIdx.x / CG, n_units = gridDim.x / CG;  // CTA pairs (CG = 2) or CTAs
  const int num_tiles = P.tiles_m * P.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], EPI_WARPS * CG);
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    async::fence_mbar_init();
    async::prefetch_tensormap(&map_a);
    async::prefetch_tensormap(&map_b);
  }
  if (warp == 1) tmem_alloc<CG, TMEM_COLS>(&sm.tmem_base);
  tc_fence_before();
  if constexpr (CG == 2) {
    async::cluster_arrive();  // barriers initialised in both CTAs before any remote use
    async::cluster_wait();
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // the even CTA's barriers, as shared::cluster addresses
  const uint32_t full0 = CG == 2 ? async::mapa(su32(&sm.full[0]), 0) : su32(&sm.full[0]);
  const uint32_t acc_empty0 = CG == 2 ? async::mapa(su32(&sm.acc_empty[0]), 0) : su32(&sm.acc_empty[0]);

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs load their own halves)
    if (lane == 0 && !P.stall) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = unit; ok && tile < num_tiles; tile += n_units) {
        const int m0 = (tile % P.tiles_m) * C::MMA_M + (int)rank * BM;
        const int n0 = (tile / P.tiles_m) * BN + (int)rank * C::B_ROWS;
        for (int kb = 0; kb < P.n_kb; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1, &sm.abort, flags, P.wait_ns)) {
            ok = false;
            break;
          }
          if (leader) mbar_expect_tx(&sm.full[stage], C::STAGE_BYTES * CG);
          const uint32_t fb = full0 + stage * 8;
          tma_load<CG>(sm.a[stage], &map_a, fb, kb * BK, m0);
          tma_load<CG>(sm.b[stage], &map_b, fb, kb * BK, n0);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        if (leader) {
          // let the copies this pair issued land before the CTA exits
          for (int i = 0; i < C::STAGES && issued > 0; ++i, --issued) {
            if (--stage < 0) {
              stage = C::STAGES - 1;
              phase ^= 1;
            }
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&sm.full[stage], phase) && global_ns() - t0 < 10000000ull) {
            }
          }
        } else {
          // this CTA's copies complete on the even CTA's barriers: give them
          // a bounded grace period instead
          const uint64_t t0 = global_ns();
          while (global_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (the even CTA issues for the pair)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t chunk_ctr = 0;
      bool ok = true;
      for (int tile = unit; ok && tile < num_tiles; tile += n_units) {
        for (int c = 0; ok && c < P.n_chunks; ++c) {
          const uint32_t buf = chunk_ctr & 1, use = chunk_ctr >> 1;
          if (!mbar_wait(&sm.acc_empty[buf], (use & 1) ^ 1, &sm.abort, flags, P.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + buf * TMEM_BUF_STRIDE;
          const int kb0 = c * CHUNK_KB, kb1 = min(P.n_kb, kb0 + CHUNK_KB);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&sm.full[stage], phase, &sm.abort, flags, P.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = su32(sm.a[stage]), b_addr = su32(sm.b[stage]);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_f16<CG>(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32),
                          F16 ? C::IDESC_F16 : C::IDESC,
                           (kb > kb0 || kk > 0) ? 1u : 0u);
            mma_commit<CG>(&sm.empty[stage]);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          mma_commit<CG>(&sm.acc_full[buf]);
          ++chunk_ctr;
        }
      }
      // wait for every MMA this thread issued before TMEM is released
      asm volatile("tcgen05.commit.cta_group::%1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       su32(&sm.drain)),
                   "n"(CG)
                   : "memory");
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(&sm.drain, 0) && global_ns() - t0 < WAIT_LIMIT_NS) {
      }
    }
  } else {
    // ---------------- epilogue warps: drain chunks, then write Y
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the BN columns
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t chunk_ctr = 0;
    bool ok = true;
    for (int tile = unit; ok && tile < num_tiles; tile += n_units) {
      const int64_t m0 = (int64_t)(tile % P.tiles_m) * C::MMA_M + (int64_t)rank * BM;
      const int64_t n0 = (int64_t)(tile / P.tiles_m) * BN;
      const int64_t m = m0 + q * 32 + lane;
      const int64_t nb = n0 + half * C::COLS;
      // the scales' L2 round trips overlap the wait for the first chunk
      float* wsw = sm.ws[warp - 2];
      __syncwarp();  // the previous tile's reads of wsw are done
      for (int i = lane; i < C::COLS; i += 32) wsw[i] = (nb + i < P.N) ? __ldg(w_scale + nb + i) : 0.0f;
      const float xs = (m < P.M) ? __ldg(x_scale + m) : 0.0f;
      __syncwarp();
      int32_t acc[C::COLS];
#pragma unroll
      for (int i = 0; i < C::COLS; ++i) acc[i] = 0;
      for (int c = 0; c < P.n_chunks; ++c) {
        const uint32_t buf = chunk_ctr & 1, use = chunk_ctr >> 1;
        // one lane waits and the warp follows its result, so the warp stays
        // converged for the .sync.aligned TMEM loads
        int got = 1;
        if (lane == 0) got = mbar_wait(&sm.acc_full[buf], use & 1, &sm.abort, flags, P.wait_ns) ? 1 : 0;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
        const uint32_t base = tmem + lane_base + buf * TMEM_BUF_STRIDE + half * C::COLS;
#pragma unroll
        for (int j = 0; j < C::COLS / 8; j += 2) {
          uint32_t r[2][8];
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (j + u < C::COLS / 8) tmem_ld8(base + (j + u) * 8, r[u]);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (j + u < C::COLS / 8) {
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[(j + u) * 8 + i] += f32_to_i32_exact(r[u][i]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 2)
            mbar_arrive_cluster(acc_empty0 + buf * 8);
          else
            async::mbar_arrive_local(&sm.acc_empty[buf]);
        }
        ++chunk_ctr;
      }
      if (!ok) break;
      if (P.tma_y) {
        // stage 32 rows x SLICE columns, then one TMA store per slice
        uint8_t* stg = sm.ystage[warp - 2];
        const int64_t row0 = m0 + q * 32;
#pragma unroll
        for (int sl = 0; sl < C::COLS / C::SLICE; ++sl) {
          if (lane == 0) async::bulk_wait_read_all();  // the previous slice has left shared memory
          __syncwarp();
#pragma unroll
          for (int g = 0; g < C::SLICE / 8; ++g) {
            const int gg = sl * (C::SLICE / 8) + g;
            const float4 w0 = *reinterpret_cast<const float4*>(wsw + gg * 8);
            const float4 w1 = *reinterpret_cast<const float4*>(wsw + gg * 8 + 4);
            const float ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(__fmul_rn(__int2float_rn(acc[gg * 8 + e]), xs), ws[e]);
            const int chunk = C::SW64 ? (g ^ ((lane >> 1) & 3)) : g;
            *reinterpret_cast<uint4*>(stg + lane * (C::SLICE * 2) + chunk * 16) = pack_bf16x8(v);
          }
          async::fence_proxy_async_smem();
          __syncwarp();
          const int64_t ns = nb + sl * C::SLICE;
          if (lane == 0 && row0 < P.M && ns < P.N) {
            async::tma_store_2d(&map_y, stg, (int)ns, (int)row0);
            async::bulk_commit();
          }
        }
        if (acc_out != nullptr && m < P.M) {
          // the exact accumulators, for callers that ask for them
#pragma unroll
          for (int g = 0; g < C::COLS / 8; ++g) {
            const int64_t n = nb + g * 8;
            if (n >= P.N) break;
            int32_t* arow = acc_out + m * P.N + n;
            if (n + 8 <= P.N && P.vec_ok) {
              st16(arow, make_uint4(acc[g * 8 + 0], acc[g * 8 + 1], acc[g * 8 + 2], acc[g * 8 + 3]));
              st16(arow + 4, make_uint4(acc[g * 8 + 4], acc[g * 8 + 5], acc[g * 8 + 6], acc[g * 8 + 7]));
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (n + e < P.N) arow[e] = acc[g * 8 + e];
            }
          }
        }
      } else if (m < P.M) {
#pragma unroll
        for (int g = 0; g < C::COLS / 8; ++g) {
          const int64_t n = nb + g * 8;
          if (n >= P.N) break;
          const float4 w0 = *reinterpret_cast<const float4*>(wsw + g * 8);
          const float4 w1 = *reinterpret_cast<const float4*>(wsw + g * 8 + 4);
          const float ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(__fmul_rn(__int2float_rn(acc[g * 8 + e]), xs), ws[e]);
          __nv_bfloat16* yrow = y + m * P.N + n;
          if (n + 8 <= P.N && P.vec_ok) {
            st16(yrow, pack_bf16x8(v));
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
    // the staged Y slices are written before the CTA's shared memory goes
    if (lane == 0) async::bulk_wait_all();
  }

  tc_fence_before();
  if constexpr (CG == 2) {
    // the peer may still touch this CTA's barriers and TMEM until both
    // CTAs are here
    async::cluster_arrive();
    async::cluster_wait();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<CG, TMEM_COLS>(tmem);
  }
}

// ------------------------------------------------------------------ host side
// 2-D bf16 tensor [rows x k] (k contiguous), box of 64 x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k, uint32_t box_rows, bool f16) {
  auto fn = async::tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)k * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Y [m x n] bf16 (n contiguous) for the epilogue's TMA stores: boxes of
// `slice` columns x 32 rows, 64-byte swizzle when a box row is 64 bytes.
bool make_map_y(CUtensorMap* map, void* y, int64_t m, int64_t n, uint32_t slice) {
  auto fn = async::tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)m};
  cuuint64_t strides[1] = {(cuuint64_t)n * 2};
  cuuint32_t box[2] = {slice, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  slice * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int CG, int BN, bool F16>
sq_status launch(const void* xq, const float* x_scale, const void* wq, const float* w_scale,
                 int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                 uint64_t wait_ns, int stall, cudaStream_t st) {
  using C = Cfg<CG, BN>;
  CUtensorMap ma, mb;
  if (!make_map(&ma, xq, m, k, BM, F16) || !make_map(&mb, wq, n, k, C::B_ROWS, F16)) return SQ_ERR_CUDA;
  auto kern = k_gemm_bf16c<CG, BN, F16>;
  const size_t smem = sizeof(Smem<CG, BN>) + 1024;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      }))
    return SQ_ERR_CUDA;
  Problem P;
  P.M = m;
  P.N = n;
  P.K = k;
  P.tiles_m = (int)((m + C::MMA_M - 1) / C::MMA_M);
  P.tiles_n = (int)((n + BN - 1) / BN);
  P.n_kb = (int)((k + BK - 1) / BK);
  P.n_chunks = (P.n_kb + CHUNK_KB - 1) / CHUNK_KB;
  P.vec_ok = (n % 8 == 0) && aligned16(y) && (acc_out == nullptr || aligned16(acc_out));
  CUtensorMap my;
  std::memset(&my, 0, sizeof(my));
  P.tma_y = (n % 8 == 0) && aligned16(y) && make_map_y(&my, y, m, n, C::SLICE) ? 1 : 0;
  P.stall = stall;
  P.wait_ns = wait_ns;
  const int tiles = P.tiles_m * P.tiles_n;
  const int units = std::min(tiles, sm_count() / CG);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * CG), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, ma, mb, my, x_scale, w_scale, static_cast<__nv_bfloat16*>(y),
                         acc_out, flags, P) != cudaSuccess)
    return SQ_ERR_CUDA;
  return launch_status();
}

// Output-channel tile for a CTA pair, 256 or 240.  Measured on B300 with
// the prefill, down_proj and Q/K/V workloads: narrower MMAs (N = 224, 192,
// 128) take nearly as long per instruction as N = 256, and a 240-wide tile
// takes about 0.985 of a 256-wide one.  The cost below is the per-pair
// time of the busiest pair (whole waves of tiles) plus 0.3 x the average
// load, which orders the three measured shapes correctly.
int choose_bn(int64_t m, int64_t n, int units, int mma_m) {
  const int64_t tiles_m = (m + mma_m - 1) / mma_m;
  auto cost = [&](int bn, double t) {
    const int64_t tiles = tiles_m * ((n + bn - 1) / bn);
    const int64_t waves = (tiles + units - 1) / units;
    return (double)waves * t + 0.3 * (double)tiles * t / units;
  };
  return cost(240, 0.985) < cost(256, 1.0) ? 240 : 256;
}

}  // namespace tc

// Tiles of 256 rows (CTA pairs) once M exceeds one 128-row tile.
int gemm_bf16c_cta_group(int64_t m) { return m > tc::BM ? 2 : 1; }

sq_status gemm_bf16c_tc(const void* xq, const float* x_scale, const void* wq, const float* w_scale,
                        int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                        uint64_t wait_ns, int stall, cudaStream_t st, bool f16) {
  using namespace tc;
  if (m > (int64_t)1 << 31 || n > (int64_t)1 << 31 || k > (int64_t)1 << 31) return SQ_ERR_UNSUPPORTED;
  const int cg = gemm_bf16c_cta_group(m);
  const int bn = cg == 1 ? 256 : choose_bn(m, n, sm_count() / 2, 2 * BM);
#define SQ_TC_LAUNCH(CG_, BN_)                                                                     \
  return f16 ? launch<CG_, BN_, true>(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, flags, wait_ns, \
                                      stall, st)                                                    \
             : launch<CG_, BN_, false>(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, flags, wait_ns, \
                                       stall, st)
  if (cg == 1) SQ_TC_LAUNCH(1, 256);
  if (bn == 240) SQ_TC_LAUNCH(2, 240);
  SQ_TC_LAUNCH(2, 256);
#undef SQ_TC_LAUNCH
}

// 1-byte codes widened to exact fp16 values (codes4_to_f16x2).  The codes of a (na bytes) and then b (nb bytes) are cut into chunks of
// kWidenChunk bytes (a's last chunk may be short, and b's); chunk c goes to
// block c mod gridDim.  One thread per block bulk-copies the block's chunks
// into a ring of kWidenStages buffers; every thread widens 8-code units of
// the current buffer and writes them to dst (16 bytes per unit, in order).
// Every wait on the ring is bounded (wait_ns); one that runs out sets
// SQ_FLAG_TIMEOUT and the block stops after its copies have landed.  stall:
// no copies are issued (the bounded waits' test; 0 on every product call).
constexpr int kWidenThreads = 256;
constexpr int kWidenChunk = 8192;
constexpr int kWidenStages = 4;
__global__ void __launch_bounds__(kWidenThreads) k_widen_codes(const uint8_t* __restrict__ a, int64_t na,
                                                               const uint8_t* __restrict__ b, int64_t nb,
                                                               uint4* __restrict__ dst, int32_t* flags,
                                                               uint64_t wait_ns, int stall) {
  __shared__ __align__(128) uint8_t ring[kWidenStages][kWidenChunk];
  __shared__ uint64_t full[kWidenStages];
  const int64_t ca = (na + kWidenChunk - 1) / kWidenChunk, cb = (nb + kWidenChunk - 1) / kWidenChunk;
  const int64_t chunks = ca + cb;
  // chunk c: its source, bytes and first output unit
  auto chunk = [&](int64_t c, const uint8_t*& src, uint32_t& bytes, int64_t& unit0) {
    const bool in_a = c < ca;
    const int64_t off = (in_a ? c : c - ca) * kWidenChunk, total = in_a ? na : nb;
    src = (in_a ? a : b) + off;
    bytes = (uint32_t)(total - off < kWidenChunk ? total - off : kWidenChunk);
    unit0 = ((in_a ? 0 : na) + off) / 8;
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWidenStages; ++s) async::mbar_init(&full[s], 1);
    async::fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = async::policy_evict_first();
  if (threadIdx.x == 0 && !stall) {
    for (int s = 0; s < kWidenStages; ++s) {
      const int64_t c = blockIdx.x + (int64_t)s * gridDim.x;
      if (c >= chunks) break;
      const uint8_t* src;
      uint32_t bytes;
      int64_t unit0;
      chunk(c, src, bytes, unit0);
      async::mbar_expect_tx(&full[s], bytes);
      async::bulk_g2s_hint(ring[s], src, bytes, &full[s], pol);
    }
  }
  int it = 0;
  bool ok = true;
  for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x, ++it) {
    const int s = it % kWidenStages;
    ok = async::mbar_wait_bounded(&full[s], (uint32_t)(it / kWidenStages) & 1u, wait_ns);
    if (__syncthreads_or(!ok)) break;
    const uint8_t* src;
    uint32_t bytes;
    int64_t unit0;
    chunk(c, src, bytes, unit0);
    const int units = (int)(bytes / 8);
#pragma unroll 4
    for (int u = threadIdx.x; u < units; u += kWidenThreads) {
      const uint2 v = *reinterpret_cast<const uint2*>(ring[s] + u * 8);
      uint32_t h[4];
      codes4_to_f16x2(v.x, h[0], h[1]);
      codes4_to_f16x2(v.y, h[2], h[3]);
      st16(dst + unit0 + u, make_uint4(h[0], h[1], h[2], h[3]));
    }
    __syncthreads();  // the buffer is read: refill it with the chunk kWidenStages steps ahead
    if (threadIdx.x == 0 && !stall) {
      const int64_t cn = c + (int64_t)kWidenStages * gridDim.x;
      if (cn < chunks) {
        const uint8_t* srcn;
        uint32_t bytesn;
        int64_t unitn;
        chunk(cn, srcn, bytesn, unitn);
        async::mbar_expect_tx(&full[s], bytesn);
        async::bulk_g2s_hint(ring[s], srcn, bytesn, &full[s], pol);
      }
    }
  }
  if (!ok && threadIdx.x == 0) {
    raise_flag(flags, SQ_FLAG_TIMEOUT);
    // let the copies this block issued land before its shared memory goes
    for (int k2 = 0; k2 < kWidenStages && !stall; ++k2) {
      const int j = it + k2;
      if (blockIdx.x + (int64_t)j * gridDim.x >= chunks) break;
      async::mbar_wait_bounded(&full[j % kWidenStages], (uint32_t)(j / kWidenStages) & 1u, 10000000ull);
    }
  }
}

// Bytes of workspace the widened operands take (X then W, fp16).
size_t gemm_widen_bytes(int64_t m, int64_t n, int64_t k) { return (size_t)(m + n) * (size_t)k * 2; }

// 1-byte codes through the tensor cores: both operands widened into the
// workspace (one pass over the codes), then the fp16 form of the GEMM.
sq_status gemm_i8_widened_tc(const void* xq, const float* x_scale, const void* wq, const float* w_scale,
                             int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                             void* workspace, uint64_t wait_ns, int stall, cudaStream_t st) {
  // bytes of codes: m * k and n * k, multiples of 16 (k % 16 == 0)
  uint4* dst = static_cast<uint4*>(workspace);
  const int64_t chunks = (m * k + kWidenChunk - 1) / kWidenChunk + (n * k + kWidenChunk - 1) / kWidenChunk;
  const int64_t blocks = std::min<int64_t>(chunks, (int64_t)sm_count() * 4);
  k_widen_codes<<<(unsigned)blocks, kWidenThreads, 0, st>>>(static_cast<const uint8_t*>(xq), m * k,
                                                            static_cast<const uint8_t*>(wq), n * k, dst,
                                                            flags, wait_ns, stall);
  const sq_status r = launch_status();
  if (r != SQ_OK) return r;
  const uint8_t* xw = static_cast<const uint8_t*>(workspace);
  return gemm_bf16c_tc(xw, x_scale, xw + (size_t)m * (size_t)k * 2, w_scale, m, n, k, y, acc_out, flags,
                       wait_ns, stall, st, true);
}

}  // namespace sq
