// gemm_tc.cu -- tensor-core BitLinear GEMM for many tokens (tcgen05, sm_103a).
//
// The video transcript on yousumm.com (BitNet b1.58 2B4T, the paragraph on
// running the model on graphics cards) describes the kernel shape: weights
// travel packed and are expanded only beside the arithmetic units, which
// multiply them with 8-bit activations.  Here packed
// ternary tiles and int8 activation tiles are staged in shared memory by TMA,
// expanded next to the tensor core into an exact MMA operand format, and
// multiplied by tcgen05.mma with the accumulator in tensor memory.
//
// Exactness.  sm_103a has no integer tcgen05 MMA, so the product runs as
// kind::f16 with fp32 accumulation.  Every ternary weight and every int8
// activation is exact in fp16, every product is an integer of magnitude
// <= 128, and every partial sum is an integer of magnitude <= 128*K < 2^24
// (K <= 131072), so every intermediate is exactly representable in fp32 and
// the accumulator equals the int32 sum bit for bit.  The test-suite checks
// this on adversarial inputs that drive |acc| to 128*K.
//
// Tile: 128 output features (MMA M, operand A = W) x BN tokens (MMA N <= 256,
// operand B = x) x 64 k per stage.  Warp roles:
//   warp 0      TMA producer: packed W box [128 rows x 16 B] and int8 x box
//               [BN rows x 64 B] into a ring of raw stages;
//   warp 1      allocates tensor memory; one thread issues the MMAs;
//   warps 2..9  convert raw stages into fp16 operands (128-byte swizzled,
//               K-major), then run the epilogue (tensor memory -> y).
//
// Within every group of 16 consecutive k both operands use the order
// p = 4i + j <-> k = 4j + i.  In that order the packed word P of 16 codes
// unpacks with (P >> 2i) & 0x03030303 (codes of k = 4j + i as bytes j), and
// a sum over k does not depend on the order, so the product is unchanged.
#include <cuda.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace bl {
namespace {

constexpr int kBM = 128;         // features per tile (MMA M)
constexpr int kBK = 64;          // k per stage
constexpr int kRawStages = 4;
constexpr int kOpStages = 3;
constexpr int kConvWarps = 8;
constexpr int kThreads = 32 * (2 + kConvWarps);
constexpr int kWRawBytes = kBM * kBK / 4;     // 2048
constexpr int kARowBytes = kBK * 2;           // 128: one fp16 row of a stage
constexpr int kAOpBytes = kBM * kARowBytes;   // 16384

struct GemmCfg {
  const float* gamma;
  const float* s;
  float* y;
  int32_t* acc;
  uint32_t* err;
  int M, N, K, BN;
  int relu2;    // epilogue applies the squared ReLU
  int nstages;  // ring depth (the GEMM on pre-expanded activations)
  int stall;    // test hook: the TMA producer issues nothing
};

// ---------------------------------------------------------------- operand expansion

// Store 16-byte unit u (0..7) of row r of a 128-byte-swizzled K-major tile at shared address `tile`.
__device__ __forceinline__ void st_sw128(uint32_t tile, int r, int u, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  const uint32_t addr = tile + (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4));
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Epilogue of one 128 x BN tile: warp w (2..9) reads tensor-memory lanes
// 32*(w%4) .. +31 (= features) and the two warps of a lane quarter take
// alternate 16-token column chunks; y = fp32(acc) * fp32(gamma / s[m]).
__device__ __forceinline__ void epilogue_store(const GemmCfg& c, uint32_t tmem, const float* tscale, int warp,
                                               int lane, int n0, int m0) {
  const int q = warp & 3;
  const int n = n0 + q * 32 + lane;
  for (int j0 = ((warp - 2) >> 2) * 16; j0 < c.BN; j0 += 32) {
    uint32_t r[16];
    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)j0, r);
    if (n < c.N) {
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int m = m0 + j0 + jj;
        if (m < c.M) {
          const float v = __uint_as_float(r[jj]);
          const int64_t o = (int64_t)m * c.N + n;
          c.y[o] = out_act(__fmul_rn(v, tscale[j0 + jj]), c.relu2);
          if (c.acc) c.acc[o] = __float2int_rn(v);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- the kernel

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                   const GemmCfg c) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = c.BN;
  const int b_op_bytes = BN * kARowBytes;
  const int x_raw_bytes = BN * kBK;
  uint8_t* op_base = smem;                                          // kOpStages x (A 16 KB | B BN*128)
  uint8_t* raw_base = op_base + kOpStages * (kAOpBytes + b_op_bytes);  // kRawStages x (W 2 KB | x BN*64)
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw_base + kRawStages * (kWRawBytes + x_raw_bytes));
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kRawStages;
  uint64_t* op_full = raw_empty + kRawStages;
  uint64_t* op_empty = op_full + kOpStages;
  uint64_t* acc_full = op_empty + kOpStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  float* tscale = reinterpret_cast<float*>(tmem_slot + 4);  // [BN]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBM;  // first feature of the tile
  const int m0 = blockIdx.y * BN;   // first token of the tile
  const int nkb = c.K / kBK;
  const uint32_t tmem_cols = BN <= 32 ? 32u : BN <= 64 ? 64u : BN <= 128 ? 128u : 256u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kConvWarps);
    }
    for (int i = 0; i < kOpStages; ++i) {
      mbar_init(&op_full[i], kConvWarps);
      mbar_init(&op_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (the whole warp, one lane issues)
    {
      int issued = 0;
      for (int kb = 0; kb < nkb && !c.stall; ++kb) {
        const int slot = kb % kRawStages;
        if (!wait_warp(&raw_empty[slot], ((uint32_t)(kb / kRawStages) & 1u) ^ 1u, c.err, abort_flag)) break;
        uint8_t* wdst = raw_base + slot * (kWRawBytes + x_raw_bytes);
        if (elect_one()) {
          mbar_arrive_expect_tx(&raw_full[slot], (uint32_t)(kWRawBytes + x_raw_bytes));
          tma_load_2d(wdst, &tmap_w, kb * (kBK / 4), n0, &raw_full[slot]);
          tma_load_2d(wdst + kWRawBytes, &tmap_x, kb * kBK, m0, &raw_full[slot]);
        }
        __syncwarp();
        issued = kb + 1;
      }
      if (*abort_flag && lane == 0) {
        for (int kb = (issued > kRawStages ? issued - kRawStages : 0); kb < issued; ++kb) {
          const uint32_t a = smem_u32(&raw_full[kb % kRawStages]), par = (uint32_t)(kb / kRawStages) & 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait_sleep(a, par, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (the whole warp, one lane issues)
    {
      const uint32_t idesc = f16_idesc(kBM, BN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int os = kb % kOpStages;
        if (!wait_warp(&op_full[os], (uint32_t)(kb / kOpStages) & 1u, c.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(op_base + os * (kAOpBytes + b_op_bytes));
        const uint32_t b_base = a_base + kAOpBytes;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_f16(tmem, sw128_desc(a_base + kk * 32), sw128_desc(b_base + kk * 32), idesc, (kb | kk) ? 1u : 0u);
          mma_commit(&op_empty[os]);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(acc_full);  // fires once every MMA issued above has completed
      __syncwarp();
    }
  } else {
    // ---------------- converters, then epilogue
    const int ct = threadIdx.x - 64;  // 0 .. 255
    pdl_wait();
    const float gamma = __ldg(c.gamma);
    for (int j = ct; j < BN; j += 32 * kConvWarps) {
      const int m = m0 + j;
      tscale[j] = m < c.M ? __fdiv_rn(gamma, __ldg(c.s + m)) : 0.0f;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConvWarps) : "memory");  // scales visible to the epilogue warps
    bool ok = true;
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int slot = kb % kRawStages, os = kb % kOpStages;
      ok = wait_flag(&op_empty[os], ((uint32_t)(kb / kOpStages) & 1u) ^ 1u, c.err, abort_flag) &&
           wait_flag(&raw_full[slot], (uint32_t)(kb / kRawStages) & 1u, c.err, abort_flag);
      if (!ok) break;
      const uint32_t wraw = smem_u32(raw_base + slot * (kWRawBytes + x_raw_bytes));
      const uint32_t xraw = wraw + kWRawBytes;
      const uint32_t aop = smem_u32(op_base + os * (kAOpBytes + b_op_bytes));
      const uint32_t bop = aop + kAOpBytes;
      // W: thread -> (row r, half h): 8 packed bytes = 32 codes = 4 swizzle units
      {
        const int r = ct >> 1, h = ct & 1;
        const uint2 pw = lds64(wraw + (uint32_t)(r * 16 + h * 8));
        uint32_t f[8];
        unpack16_f16(pw.x, f);
        st_sw128(aop, r, 4 * h + 0, f[0], f[1], f[2], f[3]);
        st_sw128(aop, r, 4 * h + 1, f[4], f[5], f[6], f[7]);
        unpack16_f16(pw.y, f);
        st_sw128(aop, r, 4 * h + 2, f[0], f[1], f[2], f[3]);
        st_sw128(aop, r, 4 * h + 3, f[4], f[5], f[6], f[7]);
      }
      // x: 16-byte chunk q of token row t -> swizzle units 2q, 2q+1
      for (int idx = ct; idx < BN * 4; idx += 32 * kConvWarps) {
        const int t = idx >> 2, q = idx & 3;
        const uint4 v = lds128(xraw + (uint32_t)(t * kBK + q * 16));
        uint32_t f[8];
        convert_x16_f16(v, f);
        st_sw128(bop, t, 2 * q, f[0], f[1], f[2], f[3]);
        st_sw128(bop, t, 2 * q + 1, f[4], f[5], f[6], f[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_empty[slot]);
        mbar_arrive(&op_full[os]);
      }
    }
    // ---- epilogue
    {
      // the issuer commits acc_full even after giving up: a thread whose own
      // waits failed, or that sees the abort flag, writes nothing
      const bool done = wait_flag(acc_full, 0u, c.err, abort_flag);
      tc_fence_after();
      if (done && ok && *abort_flag == 0u) epilogue_store(c, tmem, tscale, warp, lane, n0, m0);
      tc_fence_before();
    }
  }
  __syncthreads();
  if (warp == 1) {
    // Every MMA issued must have finished before its accumulator is freed; the
    // issuer always commits acc_full, so this completes (bounded in any case).
    const uint32_t a = smem_u32(acc_full);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(a, 0u, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
    }
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ---------------------------------------------------------------- activations expanded once per call
//
// With a workspace, the int8 activations are expanded to fp16 ONCE per call
// (by the quantisation kernel or the x_q prepass of the stream-K GEMM), in the
// operand order above (p = 4i + j within every 16 k), instead of once per
// 128-feature tile inside the GEMM; the GEMM loads the fp16 operand straight
// into its 128-byte-swizzled layout with a TMA copy.

constexpr int kX16MaxStages = 12;

// ---------------------------------------------------------------- persistent variant for large grids
//
// One CTA per SM walks the output tiles t = blockIdx.x, blockIdx.x + gridDim.x,
// ... (feature tiles fastest, so CTAs running at the same time share the
// activation tile in L2).  Two accumulators in tensor memory (2 x 256 columns)
// let eight epilogue warps drain tile t while the MMA warp and the converters
// already work on tile t+1.  Warps: 0 TMA producer, 1 MMA issuer, 2..9 W
// converters, 10..17 epilogue (two per tensor-memory lane quarter).  The ring of stages and its barriers run on
// across tiles; acc_full[b] / acc_empty[b] hand accumulator b between the MMA
// warp and the epilogue warps.

constexpr int kPEpiWarps = 8;  // two per tensor-memory lane quarter
constexpr int kPThreads = 32 * (2 + kConvWarps + kPEpiWarps);

__global__ void __launch_bounds__(kPThreads, 1)
    gemm_tc_x16_persistent_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                  const __grid_constant__ CUtensorMap tmap_x16, const GemmCfg c) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = c.BN;
  const int NS = c.nstages;
  const int b_bytes = BN * kARowBytes;
  const int stage_bytes = kAOpBytes + b_bytes + kWRawBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * stage_bytes);
  uint64_t* tma_full = bars;
  uint64_t* op_full = tma_full + kX16MaxStages;
  uint64_t* op_empty = op_full + kX16MaxStages;
  uint64_t* acc_full = op_empty + kX16MaxStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;             // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  float* tscale = reinterpret_cast<float*>(tmem_slot + 4);  // [2][BN]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = c.K / kBK;
  const int ntn = (c.N + kBM - 1) / kBM;
  const int ntiles = ntn * ((c.M + BN - 1) / BN);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&tma_full[i], 1);
      mbar_init(&op_full[i], kConvWarps);
      mbar_init(&op_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kPEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (the whole warp, one lane issues)
    {
      pdl_wait();
      int os = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok && !c.stall; t += gridDim.x) {
        const int n0 = (t % ntn) * kBM, m0 = (t / ntn) * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_warp(&op_empty[os], ph ^ 1u, c.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + os * stage_bytes;
          if (elect_one()) {
            mbar_arrive_expect_tx(&tma_full[os], (uint32_t)(b_bytes + kWRawBytes));
            tma_load_2d(st + kAOpBytes + b_bytes, &tmap_w, kb * (kBK / 4), n0, &tma_full[os]);
            tma_load_2d(st + kAOpBytes, &tmap_x16, kb * kBK, m0, &tma_full[os]);
          }
          __syncwarp();
          ++issued;
          if (++os == NS) {
            os = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && lane == 0) {
        for (int g = (issued > NS ? issued - NS : 0); g < issued; ++g) {
          const uint32_t a = smem_u32(&tma_full[g % NS]), par = (uint32_t)(g / NS) & 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait_sleep(a, par, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (the whole warp, one lane issues)
    {
      const uint32_t idesc = f16_idesc(kBM, BN);
      const uint32_t smem0 = smem_u32(smem);
      int os = 0, lt = 0;
      uint32_t par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++lt) {
        const int b = lt & 1;
        if (!wait_warp(&acc_empty[b], ((uint32_t)(lt >> 1) & 1u) ^ 1u, c.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * 256);
        // one 64-k stage; the single issuing warp's instruction stream bounds the
        // rate, so the stages are unrolled by four and op_full stands for the
        // stage's copies too (the converters waited for them before arriving)
        auto stage = [&](int kb) -> bool {
          if (!wait_warp(&op_full[os], par, c.err, abort_flag)) return false;
          tc_fence_after();
          const uint32_t a_base = smem0 + (uint32_t)(os * stage_bytes);
          const uint64_t da = sw128_desc(a_base), db = sw128_desc(a_base + kAOpBytes);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)  // 32 bytes (+2 in the address field) per MMA
              mma_f16(d, da + (uint64_t)(2 * kk), db + (uint64_t)(2 * kk), idesc, (kb | kk) ? 1u : 0u);
            mma_commit(&op_empty[os]);
          }
          __syncwarp();
          if (++os == NS) {
            os = 0;
            par ^= 1u;
          }
          return true;
        };
        int kb = 0;
#pragma unroll 1
        for (; kb + 4 <= nkb && ok; kb += 4) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (!stage(kb + u)) {
              ok = false;
              break;
            }
        }
        for (; kb < nkb && ok; ++kb)
          if (!stage(kb)) ok = false;
        if (ok && elect_one()) mma_commit(&acc_full[b]);
        __syncwarp();
      }
    }
  } else if (warp < 2 + kConvWarps) {
    // ---------------- W converters
    const int ct = threadIdx.x - 64;  // 0 .. 255
    const int r = ct >> 1, h = ct & 1;
    int os = 0;
    uint32_t par = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb) {
        if (!wait_flag(&tma_full[os], par, c.err, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t aop = smem_u32(smem + os * stage_bytes);
        const uint2 pw = lds64(aop + kAOpBytes + b_bytes + (uint32_t)(r * 16 + h * 8));
        uint32_t f[8];
        unpack16_f16(pw.x, f);
        st_sw128(aop, r, 4 * h + 0, f[0], f[1], f[2], f[3]);
        st_sw128(aop, r, 4 * h + 1, f[4], f[5], f[6], f[7]);
        unpack16_f16(pw.y, f);
        st_sw128(aop, r, 4 * h + 2, f[0], f[1], f[2], f[3]);
        st_sw128(aop, r, 4 * h + 3, f[4], f[5], f[6], f[7]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&op_full[os]);
        if (++os == NS) {
          os = 0;
          par ^= 1u;
        }
      }
    }
  } else {
    // ---------------- epilogue warps: tensor-memory lane quarter q = warp % 4
    const int et = threadIdx.x - 32 * (2 + kConvWarps);  // 0 .. 127
    const int q = warp & 3;
    pdl_wait();
    const float gamma = __ldg(c.gamma);
    int lt = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
      const int b = lt & 1;
      const int n0 = (t % ntn) * kBM, m0 = (t / ntn) * BN;
      float* ts = tscale + b * BN;
      for (int j = et; j < BN; j += 32 * kPEpiWarps) {
        const int m = m0 + j;
        ts[j] = m < c.M ? __fdiv_rn(gamma, __ldg(c.s + m)) : 0.0f;
      }
      // one barrier of the epilogue warps makes the scales visible and settles, for
      // every warp alike, whether the accumulator came (a warp whose wait gave
      // up must not leave the others at a later barrier)
      const bool got = wait_flag(&acc_full[b], (uint32_t)(lt >> 1) & 1u, c.err, abort_flag);
      uint32_t any_failed;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 2, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(any_failed)
          : "r"((uint32_t)!got), "n"(32 * kPEpiWarps)
          : "memory");
      if (any_failed) break;
      tc_fence_after();
      const int n = n0 + q * 32 + lane;
      // the two warps of a lane quarter take alternate 16-token chunks
      for (int j0 = ((warp - (2 + kConvWarps)) >> 2) * 16; j0 < BN; j0 += 32) {
        uint32_t rr[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 256 + j0), rr);
        if (n < c.N) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int m = m0 + j0 + jj;
            if (m < c.M) {
              const float v = __uint_as_float(rr[jj]);
              const int64_t o = (int64_t)m * c.N + n;
              c.y[o] = out_act(__fmul_rn(v, ts[j0 + jj]), c.relu2);
              if (c.acc) c.acc[o] = __float2int_rn(v);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    // every MMA this thread issued has finished before tensor memory is freed
    if (elect_one()) mma_commit(drain);  // the issuing lane: its MMAs are the ones tracked
    __syncwarp();
    const uint32_t a = smem_u32(drain);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(a, 0u, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
    }
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side

// Token tiles of equal size, rounded up to the MMA's N granularity of 16.
int token_tile(int64_t M, int64_t* ntiles) {
  *ntiles = (M + 255) / 256;
  const int BN = (int)((M + *ntiles - 1) / *ntiles);
  return (BN + 15) / 16 * 16;
}

}  // namespace

bool gemm_x16_persistent_serves(int64_t M, int64_t N, int num_sms) {
  int64_t ntiles = 0;
  const int BN = token_tile(M, &ntiles);
  const int64_t tiles = (N + kBM - 1) / kBM * ntiles;
  return BN >= 128 && tiles >= 2 * (int64_t)num_sms;
}


namespace {

constexpr size_t kMaxDynSmem = 227 * 1024;  // per CTA (opt-in limit)

}  // namespace

cudaError_t launch_gemm_tc_x16(const ForwardArgs& a, const void* x16, int num_sms, cudaStream_t stream) {
  int64_t ntiles = 0;
  const int BN = token_tile(a.M, &ntiles);
  const int64_t tiles = (a.N + kBM - 1) / kBM * ntiles;
  if (tiles < num_sms || BN < 128) return cudaErrorInvalidValue;  // the stream-K GEMM serves these shapes
  CUtensorMap tw, tx;
  if (!encode_u8_2d(&tw, a.Wp, (uint64_t)a.K / 4, (uint64_t)a.N, kBK / 4, kBM, 0)) return cudaErrorInvalidValue;
  if (!encode_f16_2d_sw128(&tx, x16, (uint64_t)a.K, (uint64_t)a.M, (uint32_t)BN)) return cudaErrorInvalidValue;
  // one CTA per SM, the deepest ring that fits beside [2][BN] scales
  const size_t stage = kAOpBytes + (size_t)BN * kARowBytes + kWRawBytes;
  const size_t fixed = 1024 + (3 * kX16MaxStages + 5) * 8 + 16 + (size_t)BN * 8;
  int NS = (int)((kMaxDynSmem - fixed) / stage);
  if (NS > kX16MaxStages) NS = kX16MaxStages;
  const size_t smem = fixed + (size_t)NS * stage;
  cudaError_t e =
      cudaFuncSetAttribute(gemm_tc_x16_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  GemmCfg c{a.gamma, a.s, a.y, a.acc, a.err, (int)a.M, (int)a.N, (int)a.K, BN, a.relu2 ? 1 : 0, NS,
            a.test_stall ? 1 : 0};
  const int grid = (int)(tiles < num_sms ? tiles : num_sms);
  // a programmatic dependent of the preceding kernel (the quantisation or the
  // prepass): set-up starts before it ends; the producer and the epilogue wait
  // for it (griddepcontrol.wait) before reading its output
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_x16_persistent_kernel, tw, tx, c);
}

cudaError_t launch_gemm_tc(const ForwardArgs& a, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  int64_t ntiles = 0;
  const int BN = token_tile(a.M, &ntiles);
  CUtensorMap tw, tx;
  if (!encode_u8_2d(&tw, a.Wp, (uint64_t)a.K / 4, (uint64_t)a.N, kBK / 4, kBM, 0)) return cudaErrorInvalidValue;
  if (!encode_u8_2d(&tx, a.xq, (uint64_t)a.K, (uint64_t)a.M, kBK, (uint32_t)BN, 0)) return cudaErrorInvalidValue;
  GemmCfg c{a.gamma, a.s, a.y, a.acc, a.err, (int)a.M, (int)a.N, (int)a.K, BN, a.relu2 ? 1 : 0, 0,
            a.test_stall ? 1 : 0};
  const size_t smem = 1024 + (size_t)kOpStages * (kAOpBytes + BN * kARowBytes) +
                      (size_t)kRawStages * (kWRawBytes + BN * kBK) + (2 * kRawStages + 2 * kOpStages + 1) * 8 + 16 +
                      (size_t)BN * 4;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.N + kBM - 1) / kBM), (unsigned)ntiles);
  gemm_tc_kernel<<<grid, kThreads, smem, stream>>>(tw, tx, c);
  return cudaGetLastError();
}

}  // namespace bl
