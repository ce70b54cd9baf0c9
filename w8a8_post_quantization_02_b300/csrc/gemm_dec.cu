// Step 5, decode path (at most 16 tokens): exact INT8 x INT8 GEMM that
// streams the int8 weight codes once, with the bf16 dequantizing epilogue.
//
// Source: learn-kernels.com "Quantization", paragraph 1: a decode step is
// bound by streaming the weights from memory; paragraph 2: both matmul
// operands are INT8.
//
// A CTA owns 32 output channels.  Its 16 compute warps split K: warp w
// owns codes [256 w, 256 w + 256) of every 4096-code chunk of K.  The MMA
// is mma.sync m16n8k16 with the tokens as the M side (up to 16) and the
// channels as the N side (four tiles of 8): a warp widens the tokens' codes
// of its K range to exact fp16 fragments once and reuses them for all 32
// channels, so each weight code is loaded and widened exactly once.  Warp
// 0 issues, per chunk, every warp's 2-D TMA boxes (128 codes x 32 channel
// rows and 128 codes x 16 token rows, 128-byte swizzle; rows past N or M
// and codes past K arrive as 0) on that warp's own barrier, so each warp
// starts as soon as its slice has landed.  Within a 128-code k-block, lane
// c hands codes 32c + 4j .. 32c + 4j + 3 to k16 step j (j = 0..7); the MMA
// reads them as k = 2c, 2c+1, 2c+8, 2c+9 on both operands, so every
// product still pairs a token and a channel at the same k and the sum is
// unchanged.  Products are exact in fp32 and each warp converts its sums to
// int32 after every chunk (at most 256 products per output); the warps'
// int32 sums meet in shared memory at the end and the epilogue writes Y
// (and the accumulators).  Every mbarrier wait is bounded; one that runs
// out sets SQ_FLAG_TIMEOUT.
#include <cuda_bf16.h>

#include "sq_async.cuh"

namespace sq {
namespace dec {
using namespace async;

constexpr int kChan = 32;                         // output channels per CTA (four n8 tiles)
constexpr int kKBlock = 128;                      // codes per k-block (one swizzled 128-byte box row)
constexpr int kWarps = 16;                        // compute warps, two k-blocks of every chunk each
constexpr int kChunk = 2 * kKBlock * kWarps;      // codes of K per chunk (4096)
constexpr int kThreads = 32 * (1 + kWarps);
constexpr int kWBox = kChan * kKBlock;            // bytes of one channel box (4 KiB)
constexpr int kXBox = 16 * kKBlock;               // bytes of one token box (2 KiB)
constexpr int kSlice = 2 * (kWBox + kXBox);       // bytes of one warp's slice of a chunk
constexpr int kSmem = kWarps * kSlice + 2 * kWarps * 8 + 16 + 1024;

SQ_DEVINL uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 16 int8 codes -> 8 registers of two exact fp16 values each (codes 2i and
// 2i + 1 in register i): byte u = code + 128 as the fp16 pattern 0x6400 | u
// is 1024 + u, minus 1152 exactly.
SQ_DEVINL void codes_to_f16(uint4 v, uint32_t* h) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[2 * i] = hsub2(__byte_perm(w[i], 0x64646464u, 0x4140), 0x64806480u);
    h[2 * i + 1] = hsub2(__byte_perm(w[i], 0x64646464u, 0x4342), 0x64806480u);
  }
}

SQ_DEVINL void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_dec(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
               const float* __restrict__ x_scale, const float* __restrict__ w_scale, int M, int64_t N,
               int64_t K, __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out,
               int32_t* flags, uint64_t wait_ns, int stall) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWarps * kSlice);  // [warp]: its slice landed
  uint64_t* empty = full + kWarps;                                       // [warp]: done with its slice
  int* abort_flag = reinterpret_cast<int*>(empty + kWarps);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = (int64_t)blockIdx.x * kChan;
  const int nch = (int)(N - n0 < kChan ? N - n0 : kChan);
  const int64_t nchunks = (K + kChunk - 1) / kChunk;

  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w) {
      mbar_init(&full[w], 1);
      mbar_init(&empty[w], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_w);
    prefetch_tensormap(&map_x);
  }
  __syncthreads();

  auto wait = [&](uint64_t* b, uint32_t parity) -> bool {
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
      if (mbar_try_wait(b, parity)) return true;
      if ((i & 63) == 0) {
        if (*(volatile int*)abort_flag) return false;
        if (global_ns() - t0 > wait_ns) {
          *(volatile int*)abort_flag = 1;
          raise_flag(flags, SQ_FLAG_TIMEOUT);
          return false;
        }
      }
    }
  };

  if (warp == 0) {
    // ---------------- producer: every warp's slice of every chunk, k-blocks below K only
    // (stall: none, the bounded waits' test; 0 on every product call)
    if (lane == 0 && !stall) {
      int64_t issued_to = 0;  // chunks issued
      bool ok = true;
      for (int64_t ch = 0; ok && ch < nchunks; ++ch) {
        for (int w = 0; w < kWarps; ++w) {
          const int64_t k0 = ch * kChunk + (int64_t)w * 2 * kKBlock;
          if (k0 >= K) break;  // this and later slices of the chunk lie past K
          if (!wait(&empty[w], ((uint32_t)ch & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          const int nb = K - k0 > kKBlock ? 2 : 1;
          uint8_t* sl = smem + (size_t)w * kSlice;
          mbar_expect_tx(&full[w], (uint32_t)nb * (kWBox + kXBox));
          for (int b = 0; b < nb; ++b) {
            tma_load_2d(sl + b * kWBox, &map_w, &full[w], (int)(k0 + b * kKBlock), (int)n0);
            tma_load_2d(sl + 2 * kWBox + b * kXBox, &map_x, &full[w], (int)(k0 + b * kKBlock), 0);
          }
        }
        if (ok) issued_to = ch + 1;
      }
      if (!ok || *(volatile int*)abort_flag) {
        // let the copies issued land before the CTA exits
        for (int w = 0; w < kWarps; ++w) {
          for (int64_t ch = issued_to > 0 ? issued_to - 1 : 0; ch < issued_to; ++ch) {
            if (ch * kChunk + (int64_t)w * 2 * kKBlock >= K) continue;
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&full[w], (uint32_t)ch & 1u) && global_ns() - t0 < 10000000ull) {
            }
          }
        }
      }
    }
  } else {
    // ---------------- compute warps
    const int cw = warp - 1;
    const int g = lane >> 2, c = lane & 3;
    // byte offsets of this lane's chunks 2c and 2c + 1 in a box row of
    // the 8-row atom (128-byte swizzle: chunk XOR row-within-atom, here g)
    const uint32_t off0 = (uint32_t)g * kKBlock + ((uint32_t)((2 * c) ^ g) << 4);
    const uint32_t off1 = (uint32_t)g * kKBlock + ((uint32_t)((2 * c + 1) ^ g) << 4);
    int32_t iacc[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int r = 0; r < 4; ++r) iacc[t][r] = 0;
    for (int64_t ch = 0; ch < nchunks; ++ch) {
      const int64_t k0 = ch * kChunk + (int64_t)cw * 2 * kKBlock;
      if (k0 >= K) continue;  // nothing of this chunk for this warp (no copies, no barrier phase)
      if (!__all_sync(0xFFFFFFFFu, wait(&full[cw], (uint32_t)ch & 1u))) break;
      const uint8_t* sl = smem + (size_t)cw * kSlice;
      float facc[4][4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r) facc[t][r] = 0.0f;
      const int nb = K - k0 > kKBlock ? 2 : 1;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        if (b >= nb) break;
        const uint8_t* wbox = sl + b * kWBox;
        const uint8_t* xbox = sl + 2 * kWBox + b * kXBox;
        // token fragments of the k-block: rows g and g + 8, chunks 2c and 2c + 1
        uint32_t xa[2][2][8];  // [row g / g+8][chunk]
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          codes_to_f16(*reinterpret_cast<const uint4*>(xbox + r * 8 * kKBlock + off0), xa[r][0]);
          codes_to_f16(*reinterpret_cast<const uint4*>(xbox + r * 8 * kKBlock + off1), xa[r][1]);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {  // channel tile: rows 8t + g
          uint32_t wb[2][8];
          codes_to_f16(*reinterpret_cast<const uint4*>(wbox + t * 8 * kKBlock + off0), wb[0]);
          codes_to_f16(*reinterpret_cast<const uint4*>(wbox + t * 8 * kKBlock + off1), wb[1]);
#pragma unroll
          for (int j = 0; j < 8; ++j) {  // k16 step j: codes 4(j % 4) .. +3 of chunk 2c + j / 4
            const int h = j >> 2, p = 2 * (j & 3);
            mma_f16(facc[t], xa[0][h][p], xa[1][h][p], xa[0][h][p + 1], xa[1][h][p + 1], wb[h][p],
                    wb[h][p + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_local(&empty[cw]);  // the slice is consumed
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r) iacc[t][r] += __float2int_rn(facc[t][r]);
    }
    // the warps' int32 sums meet in shared memory (every slice has been
    // consumed, so no copy is still landing in the slices)
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
    int32_t* red = reinterpret_cast<int32_t*>(smem);  // [warp][token 16][channel 32]
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int tk = g, chn = 8 * t + 2 * c;
      int32_t* r0 = red + (size_t)cw * 16 * kChan;
      r0[tk * kChan + chn] = iacc[t][0];
      r0[tk * kChan + chn + 1] = iacc[t][1];
      r0[(tk + 8) * kChan + chn] = iacc[t][2];
      r0[(tk + 8) * kChan + chn + 1] = iacc[t][3];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
    // consecutive threads take consecutive channels of one token: Y's rows
    // are written in contiguous runs
    for (int i = threadIdx.x - 32; i < 16 * kChan; i += kWarps * 32) {
      const int tk = i / kChan, chn = i % kChan;
      if (chn >= nch || tk >= M) continue;
      int32_t a = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) a += red[(size_t)w * 16 * kChan + i];
      const int64_t n = n0 + chn;
      const float v = __fmul_rn(__fmul_rn(__int2float_rn(a), x_scale[tk]), w_scale[n]);
      y[(int64_t)tk * N + n] = __float2bfloat16_rn(v);
      if (acc_out) acc_out[(int64_t)tk * N + n] = a;
    }
  }
}

// 2-D int8 tensor [rows x k] (k contiguous), boxes of 128 codes x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)k};
  cuuint32_t box[2] = {(cuuint32_t)kKBlock, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

sq_status launch(const int8_t* xq, const float* x_scale, const int8_t* wq, const float* w_scale,
                 int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                 uint64_t wait_ns, int stall, cudaStream_t st) {
  CUtensorMap mw, mx;
  if (!make_map(&mw, wq, n, k, kChan) || !make_map(&mx, xq, m, k, 16)) return SQ_ERR_CUDA;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(k_gemm_dec, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      }))
    return SQ_ERR_CUDA;
  const int64_t grid = (n + kChan - 1) / kChan;
  k_gemm_dec<<<(unsigned)grid, kThreads, kSmem, st>>>(mw, mx, x_scale, w_scale, (int)m, n, k,
                                                      static_cast<__nv_bfloat16*>(y), acc_out, flags,
                                                      wait_ns, stall);
  return launch_status();
}

}  // namespace dec

// Largest token count the decode kernel takes.
int64_t gemm_dec_max_m() { return 16; }

sq_status gemm_dec(const int8_t* xq, const float* x_scale, const int8_t* wq, const float* w_scale,
                   int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                   uint64_t wait_ns, int stall, cudaStream_t st) {
  if (m < 1 || m > 16 || n > ((int64_t)1 << 31) || k > ((int64_t)1 << 31)) return SQ_ERR_UNSUPPORTED;
  return dec::launch(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, flags, wait_ns, stall, st);
}

}  // namespace sq
