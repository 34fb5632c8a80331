// gemm_f8.cu -- tensor-core BitLinear GEMM on e4m3 operands for skinny token
// counts (tcgen05 kind::f8f6f4, sm_103a).
//
// The video transcript on yousumm.com (BitNet b1.58 2B4T, the paragraph on
// running the model on graphics cards) describes the kernel shape: weights
// travel packed and are expanded only beside the arithmetic units, which
// multiply them with 8-bit activations.  Here the packed
// ternary weights stream from HBM by TMA, are expanded next to the tensor core
// straight into tensor memory, and multiply 8-bit activation operands.
//
// Why e4m3.  At a few tokens the MMA count, not its width, sets the pace: one
// thread issues every tcgen05.mma and each takes about the same time up to an
// N of 64, so the K of one instruction decides the rate.  kind::f8f6f4 takes
// K = 32 per instruction against 16 for kind::f16, and its operands are half
// the bytes.
//
// Weights by masks.  A byte b <= 15 read as e4m3 is exactly b * 2^-9 (the
// subnormals and the first binade are evenly spaced).  So a packed word P of
// 16 codes c = W_q + 1 in {0, 1, 2} becomes weight operand bytes with two
// masks and one shift: P & 0x03030303 holds the codes k = 0, 4, 8, 12 as
// c * 2^-9, P & 0x0C0C0C0C the codes k = 1, 5, 9, 13 as 4 c * 2^-9, and the
// same two masks of P >> 4 the codes k = 2, 6, ... and 3, 7, ...  The operand
// weights are then linear in c, and the epilogue subtracts the token's sum of
// activations: sum (c - 1) x = sum c x - sum x.
//
// Exactness.  An int8 activation x is split as x = 16 h + l with h = x >> 4
// in [-8, 7] and l = x & 15 in [0, 15]; every token contributes two operand
// rows, h and l, divided by 4 at the positions whose weight byte carries 4 c,
// all exact e4m3 values.  Every product is c h 2^-9 or c l 2^-9, so each row
// of D is 2^-9 times an integer of magnitude <= 30 K <= 2^22 (K <= 131072),
// exact in the fp32 accumulator, and the epilogue forms
// acc = 16 (2^9 D_h) + 2^9 D_l - sum x in int32, exactly.
//
// Operand order.  Within every group of 16 consecutive k, both operands hold
// the k in the order p = 4 i + j <-> k = 4 j + i (word i, byte j of the
// expanded word), and a sum over k does not depend on it.
//
// Work split (stream-K).  The (output tile, 512-k block) pairs of the problem,
// tile-major, are cut into G equal contiguous ranges, one per CTA (one CTA
// per SM), so every SM streams the same number of weight bytes.  A tile whose
// k-blocks all fall in one range is finished in tensor memory.  A tile cut by
// range boundaries is reduced exactly: each contributor stores its partial
// sums (int32) to its own slot of the workspace, then adds
// its k-block count to the tile's counter; the contributor that completes the
// count adds the other slots to its own sums and writes y.
//
// Warps: 0 weight producer (TMA); 1 tensor-memory allocation and MMA issuer
// 0; 2 MMA issuer 1; 3 activation producer (bulk copies); 4..11 weight
// expansion (two per tensor-memory lane quarter, one thread per weight row);
// 12..15 epilogue (one per lane quarter).
#include <cuda.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace bl {
namespace {

constexpr int kBM = 128;                    // features per tile (MMA M)
constexpr int kKB = kX8Block;               // k per ring stage: 512
constexpr int kWStage = kBM * kKB / 4;      // 16 KB of packed weights per stage (rows of 128 bytes)
constexpr int kSub = 256;                   // k per expanded-weight slot (two per stage)
constexpr int kMaxASlots = 4;               // expanded-weight slots in tensor memory (after the accumulators)
constexpr int kACols = kSub / 4;            // 64 columns per slot: 4 e4m3 per 32-bit column
constexpr int kMaxWStages = 12, kMaxXStages = 8;
// warp roles
constexpr int kWProdWarp = 0, kMma0Warp = 1, kMma1Warp = 2, kXProdWarp = 3;
constexpr int kConvWarp0 = 4, kConvWarps = 8;  // two per tensor-memory lane quarter, each half of a slot's columns
constexpr int kEpiWarp0 = kConvWarp0 + kConvWarps, kEpiWarps = 4;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr size_t kF8SmemBudget = 220 * 1024;      // dynamic shared memory per CTA

struct F8Cfg {
  const float* gamma;
  const float* s;
  float* y;
  int32_t* acc;
  uint32_t* err;
  const uint8_t* x8;  // tiled activation operand (see x8_group_offset)
  const int32_t* sx;  // per token: x8_sum_parts(K) partial sums of its int8 activations
  int32_t* part;  // partial-sum slots: [2 * G][BN][kBM]
  uint32_t* cnt;  // arrival counters of cut tiles: [G], zero at entry
  int M, N, K, BN, nw, nx, ni, ntn, nkb, G;  // nw, nx: ring depths; ni: MMA-issuing warps (1 or 2)
  int na, acol;  // expanded-weight slots and their first tensor-memory column
  int64_t units;  // output tiles * nkb
  int relu2;
  int nsx;  // partial sums per token in sx
  int stall;  // test hook: the weight producer issues nothing
};

__device__ __forceinline__ void mma_f8_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 codes (one packed word, k = 0..15 at bits 2k) -> 16 e4m3 bytes, word i
// byte j holding code k = 4 j + i as c * 2^-9 (i even) or 4 c * 2^-9 (i odd).
__device__ __forceinline__ void expand16(uint32_t P, uint32_t* o) {
  const uint32_t T = P >> 4;
  o[0] = P & 0x03030303u;
  o[1] = P & 0x0C0C0C0Cu;
  o[2] = T & 0x03030303u;
  o[3] = T & 0x0C0C0C0Cu;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, %0;" ::"n"(32 * kEpiWarps) : "memory"); }

// Barrier of the epilogue warps that also ORs a predicate over them, so that
// every warp takes the same branch after it.
__device__ __forceinline__ bool epi_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 2, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(32 * kEpiWarps)
      : "memory");
  return r != 0;
}

// CTA whose range holds flattened k-block i: begin(c) = floor(c U / G) <= i.
__device__ __forceinline__ int cta_of(int64_t i, int64_t U, int G) { return (int)(((i + 1) * G + U - 1) / U) - 1; }

__global__ void __launch_bounds__(kThreads, 1) gemm_f8_kernel(const __grid_constant__ CUtensorMap tmap_w, const F8Cfg c) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = c.BN, NB = 2 * BN;  // MMA N: an h row and an l row per token
  const int NW = c.nw, NX = c.nx, NI = c.ni, NA = c.na;
  const int b_box = NB * 128;         // one 128-byte-wide box of the activation operand
  const int b_bytes = NB * kKB;       // a k-block's activation block: four boxes
  const int x_bytes = NB * kSub;      // one stage of the activation ring: the two boxes of a sub-block
  uint8_t* wring = smem;                        // NW x 16 KB
  uint8_t* xring = smem + NW * kWStage;         // NX x x_bytes
  uint64_t* w_full = reinterpret_cast<uint64_t*>(xring + NX * x_bytes);
  uint64_t* w_empty = w_full + kMaxWStages;     // the expansion warps
  uint64_t* x_full = w_empty + kMaxWStages;
  uint64_t* x_empty = x_full + kMaxXStages;     // the consuming issuer's commit
  uint64_t* a_full = x_empty + kMaxXStages;     // the expansion warps
  uint64_t* a_empty = a_full + kMaxASlots;      // the consuming issuer's commit
  uint64_t* acc_full = a_empty + kMaxASlots;    // [2], one commit per issuer
  uint64_t* acc_empty = acc_full + 2;           // [2], the 4 epilogue warps
  uint64_t* drain = acc_empty + 2;              // [2], one per issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* last_flag = tmem_slot + 2;
  float* tscale = reinterpret_cast<float*>(tmem_slot + 4);  // [2][kF8MaxTile]
  int* tsum = reinterpret_cast<int*>(tscale + 2 * kF8MaxTile);  // [2][kF8MaxTile]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = c.units;
  const int64_t begin = (int64_t)blockIdx.x * U / c.G, end = (int64_t)(blockIdx.x + 1) * U / c.G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], kConvWarps);
    }
    for (int i = 0; i < NX; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);
    }
    for (int i = 0; i < NA; ++i) {
      mbar_init(&a_full[i], kConvWarps);
      mbar_init(&a_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], NI);
      mbar_init(&acc_empty[b], kEpiWarps);
      mbar_init(&drain[b], 1);
    }
    *abort_flag = 0u;
    *last_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == kMma0Warp) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWProdWarp || warp == kXProdWarp) {
    // ---------------- producers (whole warps, one lane issues): the packed
    // weights (2-D TMA boxes of 128 rows x 128 B) and the activation blocks
    // (one 1-D bulk copy each)
    {
      const bool wprod = warp == kWProdWarp;
      if (!wprod) pdl_wait();  // the activation operand comes from the preceding kernel
      const int NS = wprod ? NW : NX;
      uint64_t* full = wprod ? w_full : x_full;
      uint64_t* empty = wprod ? w_empty : x_empty;
      int st = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      // (token tile mt, feature tile tn, k-block kb) of unit i, stepped without division
      const int64_t t0 = begin / c.nkb;
      int kb = (int)(begin - t0 * c.nkb), tn = (int)(t0 % c.ntn);
      int64_t mt = t0 / c.ntn;
      for (int64_t i = begin; i < end && ok && !(wprod && c.stall); ++i) {
        for (int sub = 0; sub < (wprod ? 1 : kKB / kSub); ++sub) {
          if (!wait_warp(&empty[st], ph ^ 1u, c.err, abort_flag)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            if (wprod) {
              mbar_arrive_expect_tx(&full[st], (uint32_t)kWStage);
              tma_load_2d(wring + st * kWStage, &tmap_w, kb * (kKB / 4), tn * kBM, &full[st]);
            } else {
              mbar_arrive_expect_tx(&full[st], (uint32_t)x_bytes);
              bulk_g2s(xring + st * x_bytes,
                       c.x8 + ((size_t)mt * c.nkb + kb) * (size_t)b_bytes + (size_t)sub * x_bytes, (uint32_t)x_bytes,
                       &full[st]);
            }
          }
          __syncwarp();
          ++issued;
          if (++st == NS) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (++kb == c.nkb) {
          kb = 0;
          if (++tn == c.ntn) {
            tn = 0;
            ++mt;
          }
        }
      }
      if (*abort_flag && lane == 0) {
        // let every copy this CTA started land before its shared memory goes away
        for (int g = (issued > NS ? issued - NS : 0); g < issued; ++g) {
          const uint32_t a = smem_u32(&full[g % NS]), par = (uint32_t)(g / NS) & 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait_sleep(a, par, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == kMma0Warp || warp == kMma1Warp) {
    // ---------------- MMA issuers (whole warps, one lane issues): issuer q takes
    // the slots (2 k-block + sub) with sub % NI == q, into its own accumulator;
    // the epilogue adds the issuers' sums.  The eight MMAs of a slot are unrolled.
    const int q = warp == kMma0Warp ? 0 : 1;
    if (q < NI) {
      const uint32_t idesc = f16_idesc(kBM, NB);  // format fields 0: E4M3 operands under kind::f8f6f4
      const uint64_t box_step = (uint64_t)(b_box >> 4);  // one activation box in the descriptor's address field
      int lt = 0;
      // this issuer's sub-blocks are q, q + NI, q + 2 NI, ... of the CTA's sequence: their A slots and x stages
      RingPos ap{q, 0u}, xp{q, 0u};
      bool ok = true;
      for (int64_t i = begin; i < end && ok; ++lt) {
        const int64_t t = i / c.nkb;
        const int kb0 = (int)(i - t * c.nkb);
        const int kb1 = (int)min((int64_t)c.nkb, kb0 + (end - i));
        const int b = lt & 1;
        if (!wait_warp(&acc_empty[b], ((uint32_t)(lt >> 1) & 1u) ^ 1u, c.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)((b * NI + q) * NB);
        uint32_t accum = 0u;  // the segment's first MMA overwrites the accumulator
        for (int kb = kb0; kb < kb1 && ok; ++kb) {
          for (int sub = q; sub < kKB / kSub; sub += NI) {
            const int as = ap.idx, xs = xp.idx;
            // both operands polled in one round trip (usually both ready), else waited for in turn
            const bool ready = __all_sync(0xffffffffu, mbar_try_wait(smem_u32(&x_full[xs]), xp.ph) &
                                                           mbar_try_wait(smem_u32(&a_full[as]), ap.ph)) != 0;
            if (!ready &&
                (!wait_warp(&x_full[xs], xp.ph, c.err, abort_flag) || !wait_warp(&a_full[as], ap.ph, c.err, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_col = tmem + (uint32_t)(c.acol + as * kACols);
            const uint64_t bs = sw128_desc(smem_u32(xring + xs * x_bytes));  // boxes 0, 1 of the stage
            if (elect_one()) {
              // K = 32 per MMA: +32 bytes (+2 in the address field) within a box
              mma_f8_tmem_a(d, a_col + 0, bs + 0, idesc, accum);
              mma_f8_tmem_a(d, a_col + 8, bs + 2, idesc, 1u);
              mma_f8_tmem_a(d, a_col + 16, bs + 4, idesc, 1u);
              mma_f8_tmem_a(d, a_col + 24, bs + 6, idesc, 1u);
              mma_f8_tmem_a(d, a_col + 32, bs + box_step + 0, idesc, 1u);
              mma_f8_tmem_a(d, a_col + 40, bs + box_step + 2, idesc, 1u);
              mma_f8_tmem_a(d, a_col + 48, bs + box_step + 4, idesc, 1u);
              mma_f8_tmem_a(d, a_col + 56, bs + box_step + 6, idesc, 1u);
              mma_commit(&a_empty[as]);
              mma_commit(&x_empty[xs]);
            }
            __syncwarp();
            accum = 1u;
            ap.step(NI, NA);
            xp.step(NI, NX);
          }
        }
        if (ok && elect_one()) mma_commit(&acc_full[b]);
        __syncwarp();
        i += kb1 - kb0;
      }
      // every MMA the issuing lane issued has finished before tensor memory is freed
      if (elect_one()) {
        mma_commit(&drain[q]);
        const uint32_t a = smem_u32(&drain[q]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait_sleep(a, 0u, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
      __syncwarp();
    }
  } else if (warp < kEpiWarp0) {
    // ---------------- weight expansion: thread = weight row r of the tile; the two
    // warps of a lane quarter each take one 128-k half of every slot
    const int qd = warp & 3, hf = (warp - kConvWarp0) >> 2, r = qd * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(c.acol + 32 * hf);
    const uint32_t sw = (uint32_t)(r & 7);  // 128-byte swizzle of the TMA box: chunk c of row r at c ^ (r & 7)
    int ws = 0, as = 0;
    uint32_t wph = 0, aph = 0;
    bool ok = true;
    for (int64_t i = begin; i < end && ok; ++i) {
      if (!wait_flag(&w_full[ws], wph, c.err, abort_flag)) break;
      const uint32_t wrow = smem_u32(wring + ws * kWStage) + (uint32_t)(r * 128);
      int as0 = as;
#pragma unroll
      for (int sub = 0; sub < kKB / kSub; ++sub) {
        if (!wait_flag(&a_empty[as], aph ^ 1u, c.err, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t c0 = (uint32_t)(4 * sub + 2 * hf);  // 16-byte chunks c0, c0 + 1: 128 k
        const uint4 v0 = lds128(wrow + 16u * (c0 ^ sw));
        const uint4 v1 = lds128(wrow + 16u * ((c0 + 1u) ^ sw));
        uint32_t o[32];
        expand16(v0.x, o + 0);
        expand16(v0.y, o + 4);
        expand16(v0.z, o + 8);
        expand16(v0.w, o + 12);
        expand16(v1.x, o + 16);
        expand16(v1.y, o + 20);
        expand16(v1.z, o + 24);
        expand16(v1.w, o + 28);
        tmem_st32(lane_base + (uint32_t)(as * kACols), o);
        if (++as == NA) {
          as = 0;
          aph ^= 1u;
        }
      }
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      fence_proxy_async_smem();  // this warp's reads of the stage before the next TMA write into it
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&a_full[as0]);
        mbar_arrive(&a_full[as0 + 1 == NA ? 0 : as0 + 1]);
        mbar_arrive(&w_empty[ws]);
      }
      if (++ws == NW) {
        ws = 0;
        wph ^= 1u;
      }
    }
  } else {
    // ---------------- epilogue: thread = output feature row r of the tile
    const int q = warp & 3, r = q * 32 + lane, et = threadIdx.x - 32 * kEpiWarp0;  // lane quarter q = warp % 4
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    pdl_wait();
    const float gamma = __ldg(c.gamma);
    const int first_tile = (int)(begin / c.nkb);
    int lt = 0;
    for (int64_t i = begin; i < end; ++lt) {
      const int64_t t = i / c.nkb;
      const int kb0 = (int)(i - t * c.nkb);
      const int kb1 = (int)min((int64_t)c.nkb, kb0 + (end - i));
      i += kb1 - kb0;
      const int b = lt & 1;
      const int n0 = (int)(t % c.ntn) * kBM, m0 = (int)(t / c.ntn) * BN;
      float* ts = tscale + b * kF8MaxTile;
      int* tx = tsum + b * kF8MaxTile;
      for (int j = et; j < BN; j += 32 * kEpiWarps) {
        const int m = m0 + j;
        ts[j] = m < c.M ? __fdiv_rn(gamma, __ldg(c.s + m)) : 0.0f;
        int sum = 0;
        if (m < c.M)
          for (int pc = 0; pc < c.nsx; ++pc) sum += __ldg(c.sx + (int64_t)m * c.nsx + pc);
        tx[j] = sum;
      }
      const bool got = wait_flag(&acc_full[b], (uint32_t)(lt >> 1) & 1u, c.err, abort_flag);
      if (epi_bar_or(!got)) break;  // the scales above are visible, and every warp agrees
      tc_fence_after();
      const int n = n0 + r;
      const bool whole = kb0 == 0 && kb1 == c.nkb;
      // sum c x of tokens j0 .. j0 + 15 from the h and l rows of every issuer's
      // accumulator: 16 (2^9 D_h) + 2^9 D_l, each 2^9 D an exact integer
      auto load_acc16 = [&](int j0, int (&a)[16]) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) a[jj] = 0;
        for (int qi = 0; qi < NI; ++qi) {
          uint32_t v[32];
          tmem_ld32(lane_base + (uint32_t)((b * NI + qi) * NB + 2 * j0), v);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            a[jj] += 16 * __float2int_rn(__fmul_rn(__uint_as_float(v[2 * jj]), 512.0f)) +
                     __float2int_rn(__fmul_rn(__uint_as_float(v[2 * jj + 1]), 512.0f));
        }
      };
      bool last = whole;
      const int my_slot = 2 * (int)blockIdx.x + ((int)t == first_tile ? 0 : 1);
      if (!whole) {
        // store this CTA's partial sums, then count the tile's k-blocks
        int32_t* slot = c.part + (size_t)my_slot * (BN * kBM);
        for (int j0 = 0; j0 < BN; j0 += 16) {
          int a[16];
          load_acc16(j0, a);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) slot[(j0 + jj) * kBM + r] = a[jj];
        }
        __threadfence();
        epi_bar();
        if (et == 0) {
          const int clo = cta_of(t * c.nkb, U, c.G);
          const uint32_t mine = (uint32_t)(kb1 - kb0);
          *last_flag = atomicAdd(c.cnt + clo, mine) + mine == (uint32_t)c.nkb ? 1u : 0u;
        }
        epi_bar();
        last = *last_flag != 0u;
        if (last) __threadfence();
      }
      if (last) {
        const int clo = whole ? 0 : cta_of(t * c.nkb, U, c.G), chi = whole ? -1 : cta_of((t + 1) * c.nkb - 1, U, c.G);
        for (int j0 = 0; j0 < BN; j0 += 16) {
          int a[16];
          load_acc16(j0, a);
          for (int cc = clo; cc <= chi; ++cc) {
            if (cc == (int)blockIdx.x) continue;
            const int ctile = (int)(((int64_t)cc * U / c.G) / c.nkb);  // first tile of CTA cc
            const int32_t* slot = c.part + (size_t)(2 * cc + (ctile == (int)t ? 0 : 1)) * (BN * kBM);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) a[jj] += __ldcg(slot + (j0 + jj) * kBM + r);
          }
          if (n < c.N) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int m = m0 + j0 + jj;
              if (m < c.M) {
                const int64_t o = (int64_t)m * c.N + n;
                const int v = a[jj] - tx[j0 + jj];  // sum (c - 1) x
                c.y[o] = out_act(__fmul_rn(__int2float_rn(v), ts[j0 + jj]), c.relu2);
                if (c.acc) c.acc[o] = v;
              }
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
  if (warp == kMma0Warp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- activation operand from x_q

// The tiled activation operand from x_q: CTA (c, m) writes the 16-k groups
// of 4096-k chunk c of token row m (rows past M and k past K as zeros) and
// that chunk's sum of activations; CTA (0, 0) also zeroes the arrival
// counters.  256 threads, one group each.
__global__ void __launch_bounds__(256) x8_prepass_kernel(const uint4* __restrict__ xq, int64_t M, int64_t K, int BN,
                                                         int64_t nkb, uint8_t* __restrict__ x8,
                                                         int32_t* __restrict__ sx, uint32_t* __restrict__ cnt,
                                                         int ncnt) {
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0u;
  const int64_t m = blockIdx.y, j = (int64_t)blockIdx.x * (kX8SumK / 16) + threadIdx.x;
  int sum = 0;
  if (j < nkb * (kX8Block / 16)) {
    uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
    if (m < M && j < K / 16) {
      const uint4 v = __ldg(xq + m * (K / 16) + j);
      x8_rows16(v, &hi, &lo);
      sum = sum16_i8(v);
    }
    *reinterpret_cast<uint4*>(x8 + x8_group_offset(m, 16 * j, 0, BN, nkb)) = hi;
    *reinterpret_cast<uint4*>(x8 + x8_group_offset(m, 16 * j, 1, BN, nkb)) = lo;
  }
  block_sum_store(sum, sx + m * gridDim.x + blockIdx.x);
}

}  // namespace

int gemm_f8_token_tile(int64_t M) {
  const int64_t ntm = (M + kF8MaxTile - 1) / kF8MaxTile;  // token tiles of at most 96
  return (int)(((M + ntm - 1) / ntm + 15) / 16 * 16);
}
int64_t gemm_f8_kblocks(int64_t K) { return (K + kX8Block - 1) / kX8Block; }

bool gemm_f8_serves(int64_t M, int64_t N, int64_t K) {
  (void)N;
  return M >= 1 && M <= kF8MaxTokens && K % 64 == 0;
}

namespace {

size_t x8_bytes(int64_t M, int64_t K) {
  const int BN = gemm_f8_token_tile(M);
  return (size_t)((M + BN - 1) / BN) * (size_t)(2 * BN) * (size_t)(gemm_f8_kblocks(K) * kX8Block);
}

struct F8Layout {
  uint8_t* x8;
  int32_t* part;
  uint32_t* cnt;
  int32_t* sx;
};

int64_t padded_tokens(int64_t M) {
  const int BN = gemm_f8_token_tile(M);
  return (M + BN - 1) / BN * BN;
}

F8Layout f8_layout(void* ws, int64_t M, int64_t K, int num_sms) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  F8Layout l;
  l.x8 = p;
  p += (x8_bytes(M, K) + 255) / 256 * 256;
  l.part = reinterpret_cast<int32_t*>(p);
  p += (size_t)2 * num_sms * gemm_f8_token_tile(M) * kBM * sizeof(int32_t);
  l.cnt = reinterpret_cast<uint32_t*>(p);
  p += ((size_t)num_sms * sizeof(uint32_t) + 255) / 256 * 256;
  l.sx = reinterpret_cast<int32_t*>(p);
  return l;
}

}  // namespace

size_t gemm_f8_workspace_bytes(int64_t M, int64_t K, int num_sms) {
  return (x8_bytes(M, K) + 255) / 256 * 256 + (size_t)2 * num_sms * gemm_f8_token_tile(M) * kBM * sizeof(int32_t) +
         ((size_t)num_sms * sizeof(uint32_t) + 255) / 256 * 256 +
         ((size_t)padded_tokens(M) * x8_sum_parts(K) * sizeof(int32_t) + 255) / 256 * 256;
}

cudaError_t launch_x8_prepass(const int8_t* xq, int64_t M, int64_t K, void* ws, int num_sms, cudaStream_t stream) {
  const F8Layout l = f8_layout(ws, M, K, num_sms);
  const int BN = gemm_f8_token_tile(M);
  const int64_t nkb = gemm_f8_kblocks(K);
  const dim3 grid((unsigned)x8_sum_parts(K), (unsigned)padded_tokens(M));
  x8_prepass_kernel<<<grid, kX8SumK / 16, 0, stream>>>(reinterpret_cast<const uint4*>(xq), M, K, BN, nkb, l.x8, l.sx,
                                                      l.cnt, num_sms);
  return cudaGetLastError();
}

uint32_t* f8_counters(void* ws, int64_t M, int64_t K, int num_sms) { return f8_layout(ws, M, K, num_sms).cnt; }
int32_t* f8_sums(void* ws, int64_t M, int64_t K, int num_sms) { return f8_layout(ws, M, K, num_sms).sx; }
uint8_t* f8_operand(void* ws) { return static_cast<uint8_t*>(ws); }

cudaError_t launch_gemm_f8(const ForwardArgs& a, void* ws, int num_sms, cudaStream_t stream) {
  const F8Layout l = f8_layout(ws, a.M, a.K, num_sms);
  const int BN = gemm_f8_token_tile(a.M);
  const int NB = 2 * BN;
  CUtensorMap tw;
  if (!encode_u8_2d(&tw, a.Wp, (uint64_t)a.K / 4, (uint64_t)a.N, kKB / 4, kBM, 128)) return cudaErrorInvalidValue;
  const int ntn = (int)((a.N + kBM - 1) / kBM);
  const int ntm = (int)((a.M + BN - 1) / BN);
  const int nkb = (int)gemm_f8_kblocks(a.K);
  const int64_t units = (int64_t)ntn * ntm * nkb;
  const int G = (int)(units < num_sms ? units : num_sms);
  // tensor memory: double-buffered accumulators (one per MMA-issuing warp),
  // then the expanded-weight slots
  const int NI = 4 * NB <= 256 ? 2 : 1;  // two issuers where their double-buffered accumulators fit in half
  const int acol = (2 * NI * NB + 63) / 64 * 64;
  int NA = (512 - acol) / kACols;
  if (NA > kMaxASlots) NA = kMaxASlots;
  if (NA < 2) return cudaErrorInvalidValue;
  const size_t xstage = (size_t)NB * kSub;
  int NX = (int)((96 * 1024) / xstage);  // the activation blocks come from L2: a short ring
  if (NX > kMaxXStages) NX = kMaxXStages;
  if (NX < 2) NX = 2;
  const size_t fixed = 1024 + (2 * kMaxWStages + 2 * kMaxXStages + 2 * kMaxASlots + 6) * 8 + 16 + 4 * kF8MaxTile * 4;
  int NW = (int)((kF8SmemBudget - fixed - NX * xstage) / kWStage);
  if (NW > kMaxWStages) NW = kMaxWStages;
  if (NW < 2) return cudaErrorInvalidValue;
  const size_t smem = fixed + (size_t)NW * kWStage + (size_t)NX * xstage;
  cudaError_t e = cudaFuncSetAttribute(gemm_f8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  F8Cfg c{a.gamma, a.s, a.y, a.acc, a.err, l.x8, l.sx, l.part, l.cnt, (int)a.M, (int)a.N, (int)a.K, BN, NW, NX, NI, ntn, nkb,
          G, NA, acol, units, a.relu2 ? 1 : 0, x8_sum_parts(a.K), a.test_stall ? 1 : 0};
  // a programmatic dependent of the preceding kernel (the quantisation or the
  // prepass): the weight stream and its expansion start before it ends; the
  // activation producer and the epilogue wait for it before reading its output
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_f8_kernel, tw, c);
}

}  // namespace bl
