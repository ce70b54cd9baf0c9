// Step 5, decode path (at most 16 tokens): exact INT8 x INT8 GEMM that
// streams the int8 weight codes once, with the bf16 dequantizing epilogue.
//
// Source: learn-kernels.com "Quantization", paragraph 1: a decode step is
// bound by streaming the weights from memory; paragraph 2: both matmul
// operands are INT8.
//
// A CTA owns 32 output channels and has 16 warps that split K: warp w
// owns codes [256 w, 256 w + 256) of every 4096-code chunk of K, as two
// 128-code k-blocks.  The MMA is mma.sync m16n8k16 with the tokens as the
// M side (up to 16) and the channels as the N side (four tiles of 8): a
// warp widens the tokens' codes of a k-block to exact fp16 fragments once
// and reuses them for all 32 channels, so each weight code is loaded and
// widened exactly once.  Each warp fetches its own k-blocks (one lane
// issues, per k-block, a 2-D TMA box of 128 codes x 32 channel rows and one
// of 128 codes x 16 token rows, 128-byte swizzle; rows past N or M and
// codes past K arrive as 0) into two buffers with a barrier each, and
// refetches a buffer for the next chunk as soon as it has consumed it.
// Sixteen issuing warps instead of one producer thread: a single thread
// issuing the CTA's 64 boxes took about 6 us on B300, longer than the
// weights take to stream from HBM.  Within a k-block, lane c hands codes
// 32c + 4j .. 32c + 4j + 3 to k16 step j (j = 0..7); the MMA reads them as
// k = 2c, 2c+1, 2c+8, 2c+9 on both operands, so every product still pairs a
// token and a channel at the same k and the sum is unchanged.  Products are
// exact in fp32 and each warp converts its sums to int32 after every chunk
// (at most 256 products per output); the warps' int32 sums meet in shared
// memory at the end, and each thread writes one output of Y (and of the
// accumulators) with the scales it loaded before the first copy landed.
// Every mbarrier wait is bounded; one that runs out sets SQ_FLAG_TIMEOUT.
#include <cuda_bf16.h>

#include "sq_async.cuh"

namespace sq {
namespace dec {
using namespace async;

constexpr int kChan = 32;                         // output channels per CTA (four n8 tiles)
constexpr int kKBlock = 128;                      // codes per k-block (one swizzled 128-byte box row)
constexpr int kWarps = 16;                        // warps, two k-blocks of every chunk each
constexpr int kChunk = 2 * kKBlock * kWarps;      // codes of K per chunk (4096)
constexpr int kThreads = 32 * kWarps;             // one output (token, channel) per thread at the end
constexpr int kWBox = kChan * kKBlock;            // bytes of one channel box (4 KiB)
constexpr int kXBox = 16 * kKBlock;               // bytes of one token box (2 KiB)
constexpr int kBuf = kWBox + kXBox;               // one k-block buffer: channel box, then token box
constexpr int kSlice = 2 * kBuf;                  // a warp's two buffers
constexpr int kSmem = kWarps * kSlice + 2 * kWarps * 8 + 16 + 1024;
static_assert(kThreads == 16 * kChan, "the epilogue maps threads onto 16 tokens x 32 channels");
static_assert(kWBox % 1024 == 0 && kXBox % 1024 == 0, "boxes start on 128-byte-swizzle atoms");

// 16 int8 codes -> 8 registers of two exact fp16 values each (codes 2i and
// 2i + 1 in register i), by codes4_to_f16x2.
SQ_DEVINL void codes_to_f16(uint4 v, uint32_t* h) {
  codes4_to_f16x2(v.x, h[0], h[1]);
  codes4_to_f16x2(v.y, h[2], h[3]);
  codes4_to_f16x2(v.z, h[4], h[5]);
  codes4_to_f16x2(v.w, h[6], h[7]);
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
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWarps * kSlice);  // [warp][buffer]
  int* abort_flag = reinterpret_cast<int*>(full + 2 * kWarps);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = (int64_t)blockIdx.x * kChan;
  const int nch = (int)(N - n0 < kChan ? N - n0 : kChan);
  const int64_t nchunks = (K + kChunk - 1) / kChunk;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2 * kWarps; ++b) mbar_init(&full[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_w);
    prefetch_tensormap(&map_x);
  }
  // this thread's output at the end, and its two scales, loaded now so the
  // loads overlap the weight stream
  const int out_tk = threadIdx.x / kChan, out_ch = threadIdx.x % kChan;
  const bool has_out = out_tk < M && out_ch < nch;
  float xs = 0.0f, wsc = 0.0f;
  if (has_out) {
    xs = x_scale[out_tk];
    wsc = w_scale[n0 + out_ch];
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

  // this warp's two k-block buffers; buffer h holds k-block h of the warp's
  // slice of one chunk at a time (stall: nothing is ever fetched, the
  // bounded waits' test; 0 on every product call)
  uint8_t* sl = smem + (size_t)warp * kSlice;
  uint64_t* my_full = full + 2 * warp;
  const int64_t kw = (int64_t)warp * 2 * kKBlock;  // the warp's first code in every chunk
  auto fetch = [&](int h, int64_t k0) {  // lane 0 only
    mbar_expect_tx(&my_full[h], kBuf);
    tma_load_2d(sl + h * kBuf, &map_w, &my_full[h], (int)k0, (int)n0);
    tma_load_2d(sl + h * kBuf + kWBox, &map_x, &my_full[h], (int)k0, 0);
  };
  uint32_t fetched[2] = {0u, 0u}, used[2] = {0u, 0u};  // per buffer (the same in every lane)
  for (int h = 0; h < 2; ++h) {
    if (!stall && kw + h * kKBlock < K) {
      if (lane == 0) fetch(h, kw + h * kKBlock);
      ++fetched[h];
    }
  }

  const int g = lane >> 2, c = lane & 3;
  // byte offsets of this lane's chunks 2c and 2c + 1 in a box row of the
  // 8-row atom (128-byte swizzle: chunk XOR row-within-atom, here g)
  const uint32_t off0 = (uint32_t)g * kKBlock + ((uint32_t)((2 * c) ^ g) << 4);
  const uint32_t off1 = (uint32_t)g * kKBlock + ((uint32_t)((2 * c + 1) ^ g) << 4);
  int32_t iacc[4][4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int r = 0; r < 4; ++r) iacc[t][r] = 0;
  bool ok = true;
  for (int64_t ch = 0; ok && ch < nchunks; ++ch) {
    float facc[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int r = 0; r < 4; ++r) facc[t][r] = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t k0 = ch * kChunk + kw + h * kKBlock;
      if (k0 >= K) break;  // this and every later k-block of the warp lie past K
      if (!__all_sync(0xFFFFFFFFu, wait(&my_full[h], used[h] & 1u))) {
        ok = false;
        break;
      }
      ++used[h];
      const uint8_t* wbox = sl + h * kBuf;
      const uint8_t* xbox = wbox + kWBox;
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
          const int hh = j >> 2, p = 2 * (j & 3);
          mma_f16(facc[t], xa[0][hh][p], xa[1][hh][p], xa[0][hh][p + 1], xa[1][hh][p + 1], wb[hh][p],
                  wb[hh][p + 1]);
        }
      }
      // every lane has read the buffer: refill it with the next chunk's k-block
      __syncwarp();
      const int64_t kn = k0 + kChunk;
      if (kn < K) {
        if (lane == 0) fetch(h, kn);
        ++fetched[h];
      }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int r = 0; r < 4; ++r) iacc[t][r] += __float2int_rn(facc[t][r]);
  }
  if (!ok && lane == 0) {
    // let this warp's copies in flight land before the shared memory is reused
    for (int h = 0; h < 2; ++h) {
      if (fetched[h] > used[h]) {
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(&my_full[h], used[h] & 1u) && global_ns() - t0 < 10000000ull) {
        }
      }
    }
  }
  // the warps' int32 sums meet in shared memory (every buffer has been
  // consumed, so no copy is still landing)
  __syncthreads();
  int32_t* red = reinterpret_cast<int32_t*>(smem);  // [warp][token 16][channel 32]
  {
    int32_t* r0 = red + (size_t)warp * 16 * kChan;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int chn = 8 * t + 2 * c;
      r0[g * kChan + chn] = iacc[t][0];
      r0[g * kChan + chn + 1] = iacc[t][1];
      r0[(g + 8) * kChan + chn] = iacc[t][2];
      r0[(g + 8) * kChan + chn + 1] = iacc[t][3];
    }
  }
  __syncthreads();
  // thread i: token i / 32, channel i % 32 (Y's rows written in contiguous runs)
  if (has_out) {
    int32_t a = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) a += red[(size_t)w * 16 * kChan + threadIdx.x];
    const int64_t n = n0 + out_ch;
    const float v = __fmul_rn(__fmul_rn(__int2float_rn(a), xs), wsc);
    y[(int64_t)out_tk * N + n] = __float2bfloat16_rn(v);
    if (acc_out) acc_out[(int64_t)out_tk * N + n] = a;
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
