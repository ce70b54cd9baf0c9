// Step 5, tensor-core path on 1-byte INT8 codes: exact INT8 x INT8 GEMM
// with the bf16 dequantizing epilogue, both operands read from HBM as int8.
//
// Source: learn-kernels.com "Quantization", paragraph 2: both operands of
// the matmul are INT8 and the product runs on the low-precision hardware
// path; paragraph 1: prefill is compute-bound.
//
// sm_103a's tcgen05.mma has no integer kind.  The codes stream from HBM as
// int8 (one byte per code) into shared memory by TMA; worker warps widen
// each code to an exact fp16 value (|code| <= 127 needs 7 significand
// bits) and write it in the 128-byte-swizzled K-major layout the MMA reads;
// the MMA runs as kind::f16 with both operands fp16 and fp32 accumulation
// in tensor memory.  Every product is an integer of magnitude <= 127^2 and
// every sum of at most 1024 products stays below 2^24, so the K loop is cut
// into chunks of 1024 products whose fp32 accumulators are exact integers;
// the worker warps convert each finished chunk to int32 and add it to
// running sums held in registers while the MMA fills the other of two TMEM
// accumulator buffers.
//
// Per CTA (20 warps): warp 0 issues the TMA loads of int8 k-blocks (128
// rows of A and BN/CG rows of B, 64 codes deep) into a ring of S8 stages;
// warp 1 owns TMEM and, in the even CTA, issues the MMAs; warps 2-11 each
// widen their share of every k-block into a ring of S16 fp16 stages and
// signal it on the even CTA's stage barrier, with no barrier among them, so
// each runs ahead as far as the rings allow; warps 12-19 drain each chunk's
// accumulator and, after a tile's last chunk, write Y.  The drain warps hold 128 int32
// running sums per thread, so the warpgroups trade registers (setmaxnreg):
// warps 0-11 give theirs down to 56, warps 12-19 take 152.
//   CG = 1: one CTA per SM computes 128 x BN output tiles.
//   CG = 2: a cluster of two CTAs computes 256 x BN tiles with
//     tcgen05.mma.cta_group::2; each CTA converts its own 128 rows of A and
//     BN/2 rows of B, and both CTAs' converter warps arrive on the even
//     CTA's stage barrier before the even CTA's MMAs read the pair's shared
//     memory.  Each converter thread first makes its shared-memory writes
//     visible to the async proxy (fence.proxy.async); the warp's arrive then
//     releases them at CTA scope: in the even CTA on the stage barrier the
//     MMA issuer waits on, in the odd CTA on a barrier of its own, whose
//     completion one forwarder thread acquires and passes on to the even
//     CTA with a single release at cluster scope per stage.  (With a
//     CTA-scope release there, a stress test found whole rows of the odd
//     CTA's tile read stale in 2 of 300 runs; with every converter warp
//     releasing at cluster scope the kernel ran 75 % slower.)  The MMA
//     issuer's wait keeps the CTA-scope acquire: acquiring at cluster scope
//     on every k-block measured 25-90 % slower.
// Every mbarrier wait is bounded in time; a wait that runs out sets
// SQ_FLAG_TIMEOUT, stops the CTA's loops, waits (bounded) for its own
// outstanding copies and MMAs, frees TMEM and returns.
#include "sq_tc.cuh"

namespace sq {
namespace tc8 {
using namespace tc;

#ifndef SQ_I8C_S8
#define SQ_I8C_S8 6
#endif
#ifndef SQ_I8C_S16
#define SQ_I8C_S16 4
#endif
constexpr int BM = 128;       // accumulator lanes (rows of A) per CTA
constexpr int BK = 64;        // codes per k-block: a 64-byte int8 row, a 128-byte fp16 row
constexpr int CHUNK_KB = 16;  // k-blocks per exact fp32 chunk (1024 products)
constexpr int CONV_WARPS = 10;              // warps 2-11
#ifndef SQ_I8C_PAIR
#define SQ_I8C_PAIR 1
#endif
constexpr int PAIR = SQ_I8C_PAIR;            // k-blocks a converter warp loads before storing
constexpr int EPI_WARPS = 8;                // warps 12-19
constexpr int EPI_FIRST = 2 + CONV_WARPS;
constexpr int THREADS = (2 + CONV_WARPS + EPI_WARPS) * 32;
// Registers per thread after the exchange: warpgroups 0-1 (producer, MMA,
// converters) and 2-3 (drain).  Their sum over the CTA must not exceed the
// registers the CTA was launched with (threads x the kernel's count), or
// the increase would wait forever; the host checks the built kernel's count
// against kRegsNeeded before every launch.
constexpr int REGS_LOW = 56;
constexpr int REGS_HIGH = 152;
constexpr int kRegsNeeded = EPI_FIRST * 32 * REGS_LOW + EPI_WARPS * 32 * REGS_HIGH;
static_assert(THREADS == 640 && EPI_FIRST % 4 == 0, "five warpgroups, the drain warps in the last two");
constexpr uint32_t TMEM_COLS = 512;  // two accumulator buffers at columns 0 and 256
constexpr uint32_t TMEM_BUF_STRIDE = 256;

template <int CG, int BN>
struct Cfg {
  static constexpr int B_ROWS = BN / CG;          // rows of B this CTA loads
  static constexpr int ROWS = BM + B_ROWS;         // code rows this CTA converts per k-block
  static constexpr int A8 = BM * BK;               // int8 bytes per k-block: A rows, then B rows
  static constexpr int B8 = B_ROWS * BK;
  static constexpr int A16 = BM * BK * 2;          // fp16 bytes per k-block: A rows, then B rows
  static constexpr int B16 = B_ROWS * BK * 2;
  // The int8 ring covers the copies' latency, the fp16 ring the widening
  // plus the MMAs (6 and 4 stages measured best on the prefill layer: 4/5,
  // 3/5 and 2/6 were 4-13 % slower).
  static constexpr int S8 = CG == 2 ? SQ_I8C_S8 : 3;     // int8 stages
  static constexpr int S16 = CG == 2 ? SQ_I8C_S16 : 3;   // fp16 stages
  static constexpr int VECS = ROWS * (BK / 16);    // 16-byte code vectors per k-block
  static constexpr int MMA_M = BM * CG;
  // instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
  // (format 0 in bits 7-9 and 10-12), both K-major, N >> 3 at bit 17,
  // M >> 4 at bit 24
  static constexpr uint32_t IDESC =
      (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(MMA_M >> 4) << 24);
  static constexpr int COLS = BN / 2;  // accumulator columns per drain warp
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "MMA N");
  static_assert(B_ROWS % 8 == 0, "whole 8-row swizzle atoms");
  static_assert(COLS % 8 == 0, "epilogue works in 8-column groups");
  static_assert((BM * (BK / 16)) % 32 == 0, "a warp's vectors never straddle A and B");
};

template <int CG, int BN>
struct Smem {
  using C = Cfg<CG, BN>;
  // fp16 stages: [A rows | B rows] x 128 bytes, swizzled; 1024-aligned since
  // every part is a whole number of 8-row atoms
  uint8_t f16[C::S16][C::A16 + C::B16];
  // int8 stages: [A rows | B rows] x 64 bytes, dense (as TMA writes them)
  uint8_t i8[C::S8][C::A8 + C::B8];
  uint64_t full8[C::S8];
  uint64_t empty8[C::S8];
  uint64_t full16[C::S16];     // (even CTA) both CTAs' converters finished the stage
  uint64_t conv_done[C::S16];  // (odd CTA) its converters finished the stage
  uint64_t empty16[C::S16];
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
  int stall;   // the producer issues no copies (the bounded waits' test): 0 on every product call
  uint64_t wait_ns;  // bound on every pipeline wait
};

// 16 int8 codes (one 16-byte vector, code k in byte k) -> the same 16
// integers as exact fp16 values, elements 0-7 in `lo` and 8-15 in `hi`
// (codes4_to_f16x2 on each word).
SQ_DEVINL void codes_to_f16(uint4 v, uint4& lo, uint4& hi) {
  codes4_to_f16x2(v.x, lo.x, lo.y);
  codes4_to_f16x2(v.y, lo.z, lo.w);
  codes4_to_f16x2(v.z, hi.x, hi.y);
  codes4_to_f16x2(v.w, hi.z, hi.w);
}

// Byte offset of 16-byte chunk j of row r in a K-major tile of 128-byte
// rows with the 128-byte swizzle (8-row atoms of 1024 bytes; the chunk
// index XOR-ed with the row within the atom), the layout sw128_desc names.
SQ_DEVINL uint32_t sw128_off(int r, int j) {
  return (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u + ((uint32_t)(j ^ (r & 7)) << 4);
}

// Widen one k-block.  The int8 stage is rows of 64 codes (A's 128 rows,
// then B's), the fp16 stage the same rows of 128 bytes in the swizzled
// layout.  Converter thread wt (0 .. NW-1 within its group) takes 16-byte
// vectors q = wt, wt + NW, ...: vector q is row q / 4, codes 16 (q % 4) ..
// +15, read at byte 16 q; since NW / 4 rows is a multiple of the 8-row
// swizzle atom, the row-within-atom, and so the whole destination offset up
// to a multiple of 32 NW bytes, is the same for all of a thread's vectors:
// every address is a per-thread constant plus an immediate.  A warp's 32
// vectors are eight whole 64-byte rows (conflict-free reads); per 8 lanes
// each 16-byte store hits every bank once.
struct ConvOffsets {
  uint32_t src, dst0, dst1;
};
SQ_DEVINL ConvOffsets conv_offsets(int wt) {
  const int r = wt >> 2, j = 2 * (wt & 3);
  ConvOffsets o;
  o.src = 16u * (uint32_t)wt;
  o.dst0 = sw128_off(r, j);
  o.dst1 = o.dst0 ^ 16u;  // chunk j + 1 (j even)
  return o;
}

template <int VECS, int NW>
struct ConvRegs {
  static constexpr int N = (VECS + NW - 1) / NW;  // vectors per thread per k-block
  uint4 v[N];
};

// Load this thread's vectors of the int8 stage (the stage may be refilled
// as soon as every converter has loaded it).
template <int VECS, int NW>
SQ_DEVINL void load_block(const uint8_t* src_stage, const ConvOffsets& o, int wt, ConvRegs<VECS, NW>& r) {
  const uint8_t* src = src_stage + o.src;
#pragma unroll
  for (int i = 0; i < ConvRegs<VECS, NW>::N; ++i) {
    if (VECS % NW != 0 && i == VECS / NW && wt >= VECS % NW) break;
    r.v[i] = *reinterpret_cast<const uint4*>(src + 16 * NW * i);
  }
}

// Widen the loaded vectors into the fp16 stage.
template <int VECS, int NW>
SQ_DEVINL void store_block(uint8_t* dst_stage, const ConvOffsets& o, int wt, const ConvRegs<VECS, NW>& r) {
  static_assert(NW % 32 == 0, "NW / 4 rows keep the row within its swizzle atom");
  uint8_t* d0 = dst_stage + o.dst0;
  uint8_t* d1 = dst_stage + o.dst1;
#pragma unroll
  for (int i = 0; i < ConvRegs<VECS, NW>::N; ++i) {
    if (VECS % NW != 0 && i == VECS / NW && wt >= VECS % NW) break;
    uint4 lo, hi;
    codes_to_f16(r.v[i], lo, hi);
    *reinterpret_cast<uint4*>(d0 + 32 * NW * i) = lo;
    *reinterpret_cast<uint4*>(d1 + 32 * NW * i) = hi;
  }
}

// ------------------------------------------------------------------ kernel
template <int CG, int BN>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_i8c(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const float* __restrict__ x_scale, const float* __restrict__ w_scale,
               __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out, int32_t* flags, Problem P) {
  using C = Cfg<CG, BN>;
  extern __shared__ uint8_t smem_raw[];
  Smem<CG, BN>& sm =
      *reinterpret_cast<Smem<CG, BN>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? async::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = blockIdx.x / CG, n_units = gridDim.x / CG;  // CTA pairs (CG = 2) or CTAs
  const int num_tiles = P.tiles_m * P.tiles_n;
  const int my_tiles = unit < num_tiles ? (num_tiles - unit + n_units - 1) / n_units : 0;
  const int64_t total_blocks = (int64_t)my_tiles * P.n_kb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S8; ++s) {
      mbar_init(&sm.full8[s], 1);
      mbar_init(&sm.empty8[s], CONV_WARPS);
    }
    for (int t = 0; t < C::S16; ++t) {
      mbar_init(&sm.full16[t], CG == 2 ? CONV_WARPS + 1 : CONV_WARPS);  // + the odd CTA's forwarder
      mbar_init(&sm.conv_done[t], CONV_WARPS);
      mbar_init(&sm.empty16[t], 1);
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
  const uint32_t full16_0 = CG == 2 ? async::mapa(su32(&sm.full16[0]), 0) : su32(&sm.full16[0]);
  const uint32_t acc_empty0 = CG == 2 ? async::mapa(su32(&sm.acc_empty[0]), 0) : su32(&sm.acc_empty[0]);

  if (warp < EPI_FIRST) {
  // warpgroups 0-2: producer, MMA issuer, converters
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_LOW) : "memory");
  if (warp == 0) {
    // ---------------- TMA producer: this CTA's int8 rows of A and B
    if (lane == 0 && !P.stall) {
      int64_t issued = 0;
      bool ok = true;
      int ti = 0, kb = 0;
      for (int64_t g = 0; g < total_blocks; ++g) {
        const int s = (int)(g % C::S8);
        const uint32_t use = (uint32_t)(g / C::S8);
        if (!mbar_wait(&sm.empty8[s], (use & 1) ^ 1, &sm.abort, flags, P.wait_ns)) {
          ok = false;
          break;
        }
        const int tile = unit + ti * n_units;
        const int m0 = (tile % P.tiles_m) * C::MMA_M + (int)rank * BM;
        const int n0 = (tile / P.tiles_m) * BN + (int)rank * C::B_ROWS;
        mbar_expect_tx(&sm.full8[s], C::A8 + C::B8);
        tma_load<1>(sm.i8[s], &map_a, su32(&sm.full8[s]), kb * BK, m0);
        tma_load<1>(sm.i8[s] + C::A8, &map_b, su32(&sm.full8[s]), kb * BK, n0);
        ++issued;
        if (++kb == P.n_kb) {
          kb = 0;
          ++ti;
        }
      }
      if (!ok) {
        // let this CTA's copies land before it exits
        for (int64_t g = issued - 1; g >= 0 && g >= issued - C::S8; --g) {
          const int s = (int)(g % C::S8);
          const uint32_t par = (uint32_t)(g / C::S8) & 1u;
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(&sm.full8[s], par) && global_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (the even CTA issues for the pair)
    if (lane == 0 && leader) {
      int64_t g = 0;
      uint32_t chunk_ctr = 0;
      bool ok = true;
      for (int ti = 0; ok && ti < my_tiles; ++ti) {
        for (int c = 0; ok && c < P.n_chunks; ++c) {
          const uint32_t buf = chunk_ctr & 1, use = chunk_ctr >> 1;
          if (!mbar_wait(&sm.acc_empty[buf], (use & 1) ^ 1, &sm.abort, flags, P.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + buf * TMEM_BUF_STRIDE;
          const int kb0 = c * CHUNK_KB, kb1 = min(P.n_kb, kb0 + CHUNK_KB);
          for (int kb = kb0; kb < kb1; ++kb, ++g) {
            const int t = (int)(g % C::S16);
            const uint32_t par = (uint32_t)(g / C::S16) & 1u;
            if (!mbar_wait(&sm.full16[t], par, &sm.abort, flags, P.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = su32(sm.f16[t]), b_addr = a_addr + C::A16;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_f16<CG>(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), C::IDESC,
                           (kb > kb0 || kk > 0) ? 1u : 0u);
            mma_commit<CG>(&sm.empty16[t]);
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
    } else if (CG == 2 && !leader && lane == 0) {
      // odd CTA's forwarder: once this CTA's converters have finished a
      // stage (acquired through conv_done), one arrive on the even CTA's
      // stage barrier with release at cluster scope, cumulative over those
      // writes, so they are performed for the even CTA's MMAs before the
      // arrive reaches it (the converters themselves never wait on it)
      for (int64_t g = 0; g < total_blocks; ++g) {
        const int t = (int)(g % C::S16);
        if (!mbar_wait(&sm.conv_done[t], (uint32_t)(g / C::S16) & 1u, &sm.abort, flags, P.wait_ns)) break;
        mbar_arrive_release_cluster(full16_0 + t * 8);
      }
    }
  } else {
    // ---------------- converters: every warp widens its share of every k-block
    const int wt = threadIdx.x - 64;  // 0 .. 32 * CONV_WARPS - 1
    const ConvOffsets off = conv_offsets(wt);
    // PAIR k-blocks at a time: load them all (each int8 stage freed as soon
    // as the warp holds its codes), then widen and store each once its fp16
    // stage is free; the longer independent runs hide the loads' latency.
    for (int64_t g0 = 0; g0 < total_blocks; g0 += PAIR) {
      ConvRegs<C::VECS, CONV_WARPS * 32> regs[PAIR];
      bool ok = true;
#pragma unroll
      for (int p = 0; p < PAIR; ++p) {
        const int64_t g = g0 + p;
        if (g >= total_blocks) break;
        const int s = (int)(g % C::S8);
        // one lane per warp polls the barrier; __syncwarp passes what it
        // observed (the copies' completion) on to the other lanes
        int ok_i = 1;
        if (lane == 0) ok_i = mbar_wait(&sm.full8[s], (uint32_t)(g / C::S8) & 1u, &sm.abort, flags, P.wait_ns);
        if (!__shfl_sync(0xFFFFFFFFu, ok_i, 0)) {
          ok = false;
          break;
        }
        __syncwarp();
        load_block<C::VECS, CONV_WARPS * 32>(sm.i8[s], off, wt, regs[p]);
        __syncwarp();
        if (lane == 0) async::mbar_arrive_local(&sm.empty8[s]);
      }
      if (!ok) break;
#pragma unroll
      for (int p = 0; p < PAIR; ++p) {
        const int64_t g = g0 + p;
        if (g >= total_blocks) break;
        const int t = (int)(g % C::S16);
        // the MMAs' release of the stage, passed on by __syncwarp
        int ok_i = 1;
        if (lane == 0)
          ok_i = mbar_wait(&sm.empty16[t], ((uint32_t)(g / C::S16) & 1u) ^ 1u, &sm.abort, flags, P.wait_ns);
        if (!__shfl_sync(0xFFFFFFFFu, ok_i, 0)) {
          ok = false;
          break;
        }
        __syncwarp();
        store_block<C::VECS, CONV_WARPS * 32>(sm.f16[t], off, wt, regs[p]);
        fence_proxy_async_smem();  // this thread's fp16 writes as the tensor cores will read them
        __syncwarp();
        // the even CTA's converters arrive on its stage barrier; the odd
        // CTA's on their own CTA's barrier, which its forwarder passes on
        if (lane == 0) async::mbar_arrive_local(leader ? &sm.full16[t] : &sm.conv_done[t]);
      }
      if (!ok) break;
    }
  }
  } else {
    // ---------------- warpgroups 3-4, drain warps: chunks into int32 sums, then Y
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_HIGH) : "memory");
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - EPI_FIRST) >> 2;  // which half of the BN columns
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t chunk_ctr = 0;
    bool ok = true;
    for (int ti = 0; ok && ti < my_tiles; ++ti) {
      const int tile = unit + ti * n_units;
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
      // dequantize and write Y (and the accumulators)
      const int64_t m = (int64_t)(tile % P.tiles_m) * C::MMA_M + (int64_t)rank * BM + q * 32 + lane;
      const int64_t nb = (int64_t)(tile / P.tiles_m) * BN + half * C::COLS;
      if (m < P.M) {
        const float xs = x_scale[m];
#pragma unroll
        for (int gi = 0; gi < C::COLS / 8; ++gi) {
          const int64_t n = nb + gi * 8;
          if (n >= P.N) break;
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float ws = (n + e < P.N) ? __ldg(w_scale + n + e) : 0.0f;
            v[e] = __fmul_rn(__fmul_rn(__int2float_rn(acc[gi * 8 + e]), xs), ws);
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
              st16(arow, make_uint4(acc[gi * 8 + 0], acc[gi * 8 + 1], acc[gi * 8 + 2], acc[gi * 8 + 3]));
              st16(arow + 4, make_uint4(acc[gi * 8 + 4], acc[gi * 8 + 5], acc[gi * 8 + 6], acc[gi * 8 + 7]));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (n + e < P.N) {
                yrow[e] = __float2bfloat16_rn(v[e]);
                if (acc_out) acc_out[m * P.N + n + e] = acc[gi * 8 + e];
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  if constexpr (CG == 2) {
    // the peer may still touch this CTA's barriers, shared memory and TMEM
    // until both CTAs are here
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
// 2-D int8 tensor [rows x k] (k contiguous), boxes of 64 codes x box_rows,
// no swizzle (the workers re-lay the codes out as swizzled fp16).
bool make_map_i8(CUtensorMap* map, const void* base, int64_t rows, int64_t k, uint32_t box_rows) {
  auto fn = async::tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)k};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int CG, int BN>
sq_status launch(const void* xq, const float* x_scale, const void* wq, const float* w_scale,
                 int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                 uint64_t wait_ns, int stall, cudaStream_t st) {
  using C = Cfg<CG, BN>;
  CUtensorMap ma, mb;
  if (!make_map_i8(&ma, xq, m, k, BM) || !make_map_i8(&mb, wq, n, k, C::B_ROWS)) return SQ_ERR_CUDA;
  auto kern = k_gemm_i8c<CG, BN>;
  const size_t smem = sizeof(Smem<CG, BN>) + 1024;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      }))
    return SQ_ERR_CUDA;
  // the register exchange must fit the CTA's launch allocation (see REGS_*)
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SQ_ERR_CUDA;
  if (fa.numRegs * THREADS < kRegsNeeded) return SQ_ERR_UNSUPPORTED;
  Problem P;
  P.M = m;
  P.N = n;
  P.K = k;
  P.tiles_m = (int)((m + C::MMA_M - 1) / C::MMA_M);
  P.tiles_n = (int)((n + BN - 1) / BN);
  P.n_kb = (int)((k + BK - 1) / BK);
  P.n_chunks = (P.n_kb + CHUNK_KB - 1) / CHUNK_KB;
  P.vec_ok = (n % 8 == 0) && aligned16(y) && (acc_out == nullptr || aligned16(acc_out));
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
  if (cudaLaunchKernelEx(&cfg, kern, ma, mb, x_scale, w_scale, static_cast<__nv_bfloat16*>(y),
                         acc_out, flags, P) != cudaSuccess)
    return SQ_ERR_CUDA;
  return launch_status();
}

}  // namespace tc8

// 1-byte codes on the tensor cores: one CTA per 128 x 256 tile.  The
// CTA-pair form (CG = 2, kept above) measured slower on B300 (prefill layer
// 262 us against 247 us): the odd CTA's widened tiles reach the even CTA's
// MMAs only through a cluster-scope release per stage, whose latency the
// rings do not hide.
sq_status gemm_i8c_tc(const void* xq, const float* x_scale, const void* wq, const float* w_scale,
                      int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out, int32_t* flags,
                      uint64_t wait_ns, int stall, cudaStream_t st) {
  using namespace tc8;
  if (m > (int64_t)1 << 31 || n > (int64_t)1 << 31 || k > (int64_t)1 << 31) return SQ_ERR_UNSUPPORTED;
  return launch<1, 256>(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, flags, wait_ns, stall, st);
}

}  // namespace sq
