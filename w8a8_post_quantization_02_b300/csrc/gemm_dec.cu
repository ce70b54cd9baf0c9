// Step 5, decode path (at most 16 tokens): exact INT8 x INT8 GEMM that
// streams the int8 weight codes once, with the bf16 dequantizing epilogue.
//
// Source: learn-kernels.com "Quantization", paragraph 1: a decode step is
// bound by streaming the weights from memory; paragraph 2: both matmul
// operands are INT8.
//
// A CTA owns 32 output channels (two tiles of 16) and the whole K.  The
// weight codes are [N x K] with K contiguous, so a tile's rows are long
// contiguous runs of memory: warp 0 streams them as one-dimensional bulk
// copies of whole 2 KiB row pieces (one row per lane; HBM sees contiguous
// 2 KiB reads, not 128-byte slivers), together with the tokens' code rows
// for the same K range, into a ring of shared-memory stages; each row is
// padded by 16 bytes so the readers' 16-byte loads are free of bank
// conflicts.  A stage is one channel tile x 2048 codes of K.  Warps 1-8
// each take two 128-code k-blocks of every stage: lane (g, c) loads the
// 16-byte chunks 2c and 2c + 1 of channel rows g, g + 8 and token rows g
// (and g + 8), widens them to exact fp16 (as the int8-operand tensor-core
// kernel does) and issues mma.sync m16n8k16 with the channels as the M side
// and the tokens as the N side.  Lane c hands codes 32c + 4j .. 32c + 4j + 3
// of a k-block to k16 step j (j = 0..7); the MMA reads them as k = 2c,
// 2c+1, 2c+8, 2c+9 on both operands, so every product still pairs a channel
// and a token at the same k and the sum is unchanged.  Products are exact in
// the fp32 accumulators and every warp converts them to int32 after at most
// 1024 products per output (sums stay below 2^24).  The warps' int32 sums
// meet in shared memory at the end and the epilogue writes Y (and the
// accumulators).  Every mbarrier wait is bounded; one that runs out sets
// SQ_FLAG_TIMEOUT.
#include <cuda_bf16.h>

#include "sq_async.cuh"

namespace sq {
namespace dec {
using namespace async;

constexpr int kChan = 32;                        // output channels per CTA (two tiles of 16)
constexpr int kKBlock = 128;                     // codes per k-block
constexpr int kComputeWarps = 8;                 // two k-blocks of every stage each
constexpr int kKC = 2 * kKBlock * kComputeWarps; // codes of K per stage (2048)
constexpr int kRow = kKC + 16;                   // padded shared-memory row
constexpr int kThreads = 32 * (1 + kComputeWarps);
constexpr int kStages = 3;

template <int NT>  // token tiles of 8: M <= 8 * NT
struct Cfg {
  static constexpr int TOK = 8 * NT;
  static constexpr int ROWS = 16 + TOK;                     // channel rows, then token rows
  static constexpr int STAGE = ROWS * kRow;
  static constexpr int SMEM = kStages * STAGE + 2 * kStages * 8 + 16;
};

SQ_DEVINL uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 16 int8 codes -> 8 registers of two exact fp16 values each (codes 2i and
// 2i + 1 in register i): byte u = code + 128 as the fp16 pattern 0x6400 | u
// is 1024 + u, minus 1152 exactly.
SQ_DEVINL void codes_to_f16(uint4 v, uint32_t (&h)[8]) {
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

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_dec(const int8_t* __restrict__ xq, const float* __restrict__ x_scale,
               const int8_t* __restrict__ wq, const float* __restrict__ w_scale, int M, int64_t N,
               int64_t K, __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out,
               int32_t* flags, uint64_t wait_ns, int stall) {
  using C = Cfg<NT>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * C::STAGE);
  uint64_t* empty = full + kStages;
  int* abort_flag = reinterpret_cast<int*>(empty + kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = (int64_t)blockIdx.x * kChan;
  const int nch = (int)(N - n0 < kChan ? N - n0 : kChan);
  const int64_t nkc = (K + kKC - 1) / kKC;   // K pieces per channel tile
  const int64_t units = 2 * nkc;             // stages: tile 0's pieces, then tile 1's

  // rows no copy ever writes (channels beyond N, tokens beyond M) read as 0
  for (int i = threadIdx.x; i < kStages * C::ROWS; i += kThreads) {
    const int s = i / C::ROWS, r = i % C::ROWS;
    const bool never = r < 16 ? (r >= nch || 16 + r >= nch) : (r - 16 >= M);
    // a channel row r holds channel r of tile 0 and channel 16 + r of tile 1:
    // zero it if either is missing (the copies rewrite the rows that exist)
    if (never) {
      uint4* row = reinterpret_cast<uint4*>(smem + (size_t)s * C::STAGE + (size_t)r * kRow);
      for (int q = 0; q < kKC / 16; ++q) row[q] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kComputeWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
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
    // ---------------- producer: lane i < 16 copies channel row i of the
    // tile, lane 16 + i token row i, each a contiguous piece of K
    // (stall: none, the bounded waits' test; 0 on every product call)
    const uint64_t pol = policy_evict_first();  // the weight codes are read once
    int64_t issued = 0;
    for (int64_t u = 0; u < units && !stall; ++u) {
      const int s = (int)(u % kStages);
      int ok = 1;
      if (lane == 0) ok = wait(&empty[s], ((uint32_t)(u / kStages) & 1u) ^ 1u) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      const int tile = (int)(u / nkc);
      const int64_t k0 = (u % nkc) * kKC;
      const uint32_t kb = (uint32_t)(K - k0 < kKC ? K - k0 : kKC);  // a multiple of 16
      const int rows_w = max(0, min(16, nch - 16 * tile));
      if (lane == 0) mbar_expect_tx(&full[s], kb * (uint32_t)(rows_w + M));
      __syncwarp();
      uint8_t* st = smem + (size_t)s * C::STAGE;
      if (lane < rows_w)
        bulk_g2s_hint(st + (size_t)lane * kRow, wq + (n0 + 16 * tile + lane) * K + k0, kb, &full[s], pol);
      else if (lane >= 16 && lane - 16 < M)
        bulk_g2s(st + (size_t)lane * kRow, xq + (int64_t)(lane - 16) * K + k0, kb, &full[s]);
      ++issued;
    }
    if (lane == 0 && *(volatile int*)abort_flag) {
      // let the copies issued land before the CTA exits
      for (int64_t u = issued - 1; u >= 0 && u >= issued - kStages; --u) {
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(&full[u % kStages], (uint32_t)(u / kStages) & 1u) &&
               global_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else {
    // ---------------- compute warps
    const int w8 = warp - 1;
    const int g = lane >> 2, c = lane & 3;
    int32_t iacc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) iacc[mt][nt][r] = 0;
    bool ok = true;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      float facc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) facc[nt][r] = 0.0f;
      int pending = 0;  // products per output in facc since the last conversion
      for (int64_t kc = 0; ok && kc < nkc; ++kc) {
        const int64_t u = mt * nkc + kc;
        const int s = (int)(u % kStages);
        if (!__all_sync(0xFFFFFFFFu, wait(&full[s], (uint32_t)(u / kStages) & 1u))) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + (size_t)s * C::STAGE;
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int kblk = 2 * w8 + bb;
          const int64_t valid = K - kc * kKC - kblk * kKBlock;  // codes of this k-block below K
          if (valid <= 0) continue;
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // chunk 2c + h: k16 steps 4h .. 4h + 3
            const int byte = kblk * kKBlock + (2 * c + h) * 16;
            const bool on = (2 * c + h) * 16 < valid;  // stale bytes past K read as zeros
            uint32_t wa[2][8], xb[NT][8];
#pragma unroll
            for (int r = 0; r < 2; ++r)  // channel rows g, g + 8 of the tile
              codes_to_f16(on ? *reinterpret_cast<const uint4*>(st + (size_t)(g + 8 * r) * kRow + byte)
                              : make_uint4(0u, 0u, 0u, 0u), wa[r]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)  // token rows g, g + 8
              codes_to_f16(on ? *reinterpret_cast<const uint4*>(st + (size_t)(16 + g + 8 * nt) * kRow + byte)
                              : make_uint4(0u, 0u, 0u, 0u), xb[nt]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_f16(facc[nt], wa[0][2 * j], wa[1][2 * j], wa[0][2 * j + 1], wa[1][2 * j + 1],
                        xb[nt][2 * j], xb[nt][2 * j + 1]);
          }
          pending += kKBlock;
          if (pending == 1024) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                iacc[mt][nt][r] += __float2int_rn(facc[nt][r]);
                facc[nt][r] = 0.0f;
              }
            pending = 0;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_local(&empty[s]);  // done with the stage
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) iacc[mt][nt][r] += __float2int_rn(facc[nt][r]);
    }
    // the warps' int32 sums meet in shared memory (the ring is idle once
    // every warp is past its loop: all copies have landed and been read)
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory");
    int32_t* red = reinterpret_cast<int32_t*>(smem);  // [warp][channel 32][token TOK]
    constexpr int TOK = C::TOK;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int ch = 16 * mt + g, tk = 8 * nt + 2 * c;
        int32_t* r0 = red + (size_t)w8 * kChan * TOK;
        r0[ch * TOK + tk] = iacc[mt][nt][0];
        r0[ch * TOK + tk + 1] = iacc[mt][nt][1];
        r0[(ch + 8) * TOK + tk] = iacc[mt][nt][2];
        r0[(ch + 8) * TOK + tk + 1] = iacc[mt][nt][3];
      }
    asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory");
    // consecutive threads take consecutive channels of one token: Y's rows
    // are written in contiguous runs
    for (int i = threadIdx.x - 32; i < kChan * TOK; i += kComputeWarps * 32) {
      const int tk = i / kChan, ch = i % kChan;
      if (ch >= nch || tk >= M) continue;
      int32_t a = 0;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) a += red[(size_t)w * kChan * TOK + ch * TOK + tk];
      const int64_t n = n0 + ch;
      const float v = __fmul_rn(__fmul_rn(__int2float_rn(a), x_scale[tk]), w_scale[n]);
      y[(int64_t)tk * N + n] = __float2bfloat16_rn(v);
      if (acc_out) acc_out[(int64_t)tk * N + n] = a;
    }
  }
}

template <int NT>
sq_status launch(const int8_t* xq, const float* x_scale, const int8_t* wq, const float* w_scale,
                 int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                 uint64_t wait_ns, int stall, cudaStream_t st) {
  auto kern = k_gemm_dec<NT>;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<NT>::SMEM);
      }))
    return SQ_ERR_CUDA;
  const int64_t grid = (n + kChan - 1) / kChan;
  kern<<<(unsigned)grid, kThreads, Cfg<NT>::SMEM, st>>>(xq, x_scale, wq, w_scale, (int)m, n, k,
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
  if (m <= 8) return dec::launch<1>(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, flags, wait_ns, stall, st);
  return dec::launch<2>(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, flags, wait_ns, stall, st);
}

}  // namespace sq
