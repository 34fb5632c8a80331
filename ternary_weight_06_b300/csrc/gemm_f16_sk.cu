// gemm_f16_sk.cu -- tensor-core BitLinear GEMM for many tokens: the packed
// ternary weights are expanded straight into tensor memory, the work is split
// evenly over all SMs (stream-K), and pairs of SMs share the activation
// stream by cluster multicast; tcgen05 kind::f16, sm_103a.
//
// The video transcript on yousumm.com (BitNet b1.58 2B4T, the paragraph on
// running the model on graphics cards) describes the kernel shape: weights
// travel packed and are expanded only beside the arithmetic units, which
// multiply them with 8-bit activations.  Here the packed weights are read
// next to the tensor core, expanded, and multiply the fp16 image of the int8
// activations.
//
// Exactness.  As in every tensor-core path here: ternary weights and int8
// activations are exact in fp16, every product is an integer of magnitude
// <= 128, every partial sum an integer of magnitude <= 128 K <= 2^24, exact
// in the fp32 accumulator; a tile cut between SMs adds integer-valued fp32
// partials, exact in any order.
//
// Operands.  A = the weights, 128 output features x 16 k per MMA, expanded by
// the converter warps into slots of tensor memory (32 columns per 64 k:
// column c of a 16-k group holds the fp16 pair of positions 2c, 2c + 1); the
// converter threads read their own row's packed bytes with 16-byte loads, one
// 512-k unit ahead.  B = the activations as fp16 (the GEMM operand written by
// the quantisation kernel or the x_q prepass: within every 16-k group the
// positions p = 4 i + j hold k = 4 j + i, the order in which a packed word of
// 16 codes unpacks), BN tokens x 64 k per stage, loaded by TMA with the
// 128-byte swizzle into a ring in shared memory.
//
// Pairs.  The two CTAs of a cluster take adjacent feature tiles of the same
// token tile and walk the same k-blocks in step, so they need the same
// activation stages: each issues every other stage, multicast into both
// CTAs' shared memory.  That halves the activation copies each SM issues and
// the L2 requests behind them (a copy engine keeps only a few copies in
// flight, and their latency grows with the load).  Every CTA arms its own
// full barrier for every stage; a stage is free again once both CTAs' MMAs
// are done with it (both issuers commit to both CTAs' done barriers).
//
// One wait and one commit per stage on the MMA thread: the expanding warps
// wait for the stage's activations before they report its A slot full, so
// "A full" implies "B landed"; the stage's done barrier frees both the
// activation slot (for the producers) and the A slot of the stage (for the
// expanding warps, which reuse it NA stages later).
//
// Work split (stream-K).  The (pair of output tiles, 512-k block) units,
// tile-major, are cut into C equal contiguous ranges, one per cluster (one
// CTA per SM).  A tile whose k-blocks all fall in one range is finished in
// tensor memory; a tile cut by range boundaries is reduced exactly: each
// contributor stores its partial sums to its own slot of the workspace and
// adds its k-block count to the tile's counter; the contributor that
// completes the count adds the other slots to its own sums and writes y.
//
// Warps: 0 activation producer 0; 1 tensor-memory allocation and the MMA
// issuer; 2..9 weight expansion (thread = weight row; the four warps of set h
// expand the stages with sequence number = h mod 2); 10..17 epilogue (two
// per tensor-memory lane quarter, alternate 16-token chunks); 18 activation
// producer 1 (producer p arms the stages with sequence number = p mod 2).
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace bl {
namespace {

constexpr int kBM = 128;                 // features per tile (MMA M)
constexpr int kKB = 512;                 // k per stream-K unit
constexpr int kBK = 64;                  // k per activation stage and per expanded-weight slot
constexpr int kChunks = kKB / kBK;       // 8 activation stages per unit
constexpr int kRowB = kBK * 2;           // 128 B: one token's fp16 activations of a stage
constexpr int kACols = kBK / 2;          // 32 tensor-memory columns per expanded-weight slot
constexpr int kMaxXStages = 12, kMaxASlots = 8;
constexpr int kMmaWarp = 1, kConv0 = 2, kConvWarps = 8, kEpi0 = kConv0 + kConvWarps, kEpiWarps = 8;
constexpr int kXProducers = 2, kXProdWarp1 = kEpi0 + kEpiWarps;  // producers: warp 0, then warps kXProdWarp1 ..
constexpr int kThreads = 32 * (kXProdWarp1 + kXProducers - 1);
constexpr int kPair = 2;                  // CTAs per cluster
constexpr size_t kSmemBudget = 220 * 1024;
constexpr size_t kSmemFloor = 120 * 1024;  // one CTA per SM: the CTA holds all 512 tensor-memory columns

struct SkCfg {
  const uint8_t* Wp;  // packed weights [N][K / 4]
  const float* gamma;
  const float* s;
  float* y;
  int32_t* acc;
  uint32_t* err;
  float* part;    // partial-sum slots: [2 * G][BN][kBM]
  uint32_t* cnt;  // arrival counters of cut tiles: [G], zero at entry
  int M, N, K, BN, nx, na, acc_stride, acol, ntn, ntp, nkb, C;  // ntp: feature-tile pairs; C: clusters
  int64_t units;  // token tiles * ntp * nkb
  int relu2;
  int stall;  // test hook: the converters expand nothing
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, %0;" ::"n"(32 * kEpiWarps) : "memory"); }

// Barrier of the epilogue warps that also ORs a predicate over them.
__device__ __forceinline__ bool epi_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 2, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(32 * kEpiWarps)
      : "memory");
  return r != 0;
}

// Cluster whose range holds flattened unit i: begin(c) = floor(c U / C) <= i.
__device__ __forceinline__ int cluster_of(int64_t i, int64_t U, int C) { return (int)(((i + 1) * C + U - 1) / U) - 1; }

// 64-k activation stages of 512-k block kb (the last block of a row may be short).
__device__ __forceinline__ int unit_chunks(int kb, int K) { return min(kChunks, (K - kb * kKB) / kBK); }

// After an abort: waits (bounded) for the phases this producer armed on the
// full barriers to complete, so that no copy lands in shared memory that has
// gone away.  The producer armed the stages g = p, p + P, ... < armed_end of
// a ring of n slots, n a multiple of P; stages before the last n / P were
// consumed before their slots were armed again.
__device__ __forceinline__ void drain_ring(uint64_t* full, int n, int p, int P, int64_t armed_end) {
  int64_t g0 = armed_end - n;
  if (g0 < p) g0 = p;
  g0 = p + (g0 - p + P - 1) / P * P;
  for (int64_t g = g0; g < armed_end; g += P) {
    const uint32_t a = smem_u32(&full[g % n]), par = (uint32_t)(g / n) & 1u;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(a, par, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) gemm_f16_sk_kernel(const __grid_constant__ CUtensorMap tmap_x16,
                                                                  const SkCfg c) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = c.BN, NX = c.nx, NA = c.na;
  const int x_bytes = BN * kRowB;  // one activation stage (a multiple of 1024)
  uint8_t* xring = smem;
  uint64_t* x_full = reinterpret_cast<uint64_t*>(xring + NX * x_bytes);
  uint64_t* done = x_full + kMaxXStages;      // both CTAs' MMA commits of the stage
  uint64_t* a_full = done + kMaxXStages;      // the 4 converter warps of a set
  uint64_t* acc_full = a_full + kMaxASlots;   // [2]
  uint64_t* acc_empty = acc_full + 2;         // [2], the epilogue warps
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* last_flag = tmem_slot + 2;
  float* tscale = reinterpret_cast<float*>(tmem_slot + 4);  // [2][BN]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rho = (int)cluster_rank(), cl = (int)blockIdx.x / kPair;  // rank in the pair, cluster index
  const int64_t U = c.units;
  const int64_t begin = (int64_t)cl * U / c.C, end = (int64_t)(cl + 1) * U / c.C;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NX; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&done[i], kPair);
    }
    for (int i = 0; i < NA; ++i) mbar_init(&a_full[i], kConvWarps / 2);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    *last_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // both CTAs' barriers are initialised before any copy or commit reaches them
  cluster_sync_all();

  if (warp == 0 || warp >= kXProdWarp1) {
    // ---------------- activation producers (whole warps, one lane issues):
    // producer p arms the stages with sequence number = p mod kXProducers;
    // the copy of stage q (the box [BN x 64 fp16], multicast to both CTAs) is
    // issued by the CTA of rank q % 2
    const int p = warp == 0 ? 0 : warp - kXProdWarp1 + 1;
    pdl_wait();  // the activation operand comes from the preceding kernel
    const int64_t t0 = begin / c.nkb;
    int kb = (int)(begin - t0 * c.nkb);
    int64_t mt = t0 / c.ntp, gsq = 0;  // token tile; sequence number of the next stage
    int ntp_i = (int)(t0 - mt * c.ntp);
    RingPos sr{0, 0u};
    sr.step(p, NX);
    bool ok = true;
    for (int64_t i = begin; i < end && ok; ++i) {
      const int nch = unit_chunks(kb, c.K);
      for (int g = 0; g < nch; ++g, ++gsq) {
        if ((int)(gsq % kXProducers) != p) continue;
        if (!wait_warp(&done[sr.idx], sr.ph ^ 1u, c.err, abort_flag)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&x_full[sr.idx], (uint32_t)x_bytes);
          if ((int)(gsq % kPair) == rho)
            tma_load_2d_mc(xring + sr.idx * x_bytes, &tmap_x16, kb * kKB + g * kBK, (int)(mt * BN), &x_full[sr.idx],
                           (uint16_t)((1u << kPair) - 1u));
        }
        __syncwarp();
        sr.step(kXProducers, NX);
      }
      if (++kb == c.nkb) {
        kb = 0;
        if (++ntp_i == c.ntp) {
          ntp_i = 0;
          ++mt;
        }
      }
    }
    if (*abort_flag && lane == 0) drain_ring(x_full, NX, p, kXProducers, gsq);
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (the whole warp, one lane issues): four MMAs
    // of 16 k per 64-k stage into accumulator b
    const uint32_t idesc = f16_idesc(kBM, BN);
    const uint32_t a_col0 = tmem + (uint32_t)c.acol;
    const uint64_t bd0 = sw128_desc(smem_u32(xring));  // stage s: + s * x_bytes / 16 in the address field
    const int xstep = x_bytes >> 4;
    int lt = 0;
    RingPos xr{0, 0u}, ar{0, 0u};
    bool ok = true;
    for (int64_t i = begin; i < end && ok; ++lt) {
      const int64_t t = i / c.nkb;
      const int kb0 = (int)(i - t * c.nkb);
      const int kb1 = (int)min((int64_t)c.nkb, kb0 + (end - i));
      const int b = lt & 1;
      if (!wait_warp(&acc_empty[b], ((uint32_t)(lt >> 1) & 1u) ^ 1u, c.err, abort_flag)) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(b * c.acc_stride);
      uint32_t accum = 0u;  // the segment's first MMA overwrites the accumulator
      // one 64-k stage: the single issuing warp's instruction stream, not the
      // tensor core, bounds the rate, so addresses advance by addition and the
      // usual eight-stage unit is unrolled
      auto stage = [&]() -> bool {
        // a_full implies x_full: the expanding warps waited for the stage's activations
        if (!wait_warp(&a_full[ar.idx], ar.ph, c.err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t a_col = a_col0 + (uint32_t)(ar.idx * kACols);
        const uint64_t bd = bd0 + (uint64_t)(xr.idx * xstep);
        if (elect_one()) {
          // 16 k per MMA: 8 columns of A, 32 bytes (+2 in the address field) of B
          mma_f16_tmem_a(d, a_col + 0, bd + 0, idesc, accum);
          mma_f16_tmem_a(d, a_col + 8, bd + 2, idesc, 1u);
          mma_f16_tmem_a(d, a_col + 16, bd + 4, idesc, 1u);
          mma_f16_tmem_a(d, a_col + 24, bd + 6, idesc, 1u);
          mma_commit_mc(&done[xr.idx], (uint16_t)((1u << kPair) - 1u));  // the stage, in both CTAs
        }
        __syncwarp();
        accum = 1u;
        xr.step(1, NX);
        ar.step(1, NA);
        return true;
      };
      // two stages' operands, checked together: both are usually ready already, so
      // one round trip of polls serves both; otherwise each is waited for in turn
      auto ready2 = [&]() -> bool {
        RingPos a2 = ar;
        a2.step(1, NA);
        const bool both = mbar_try_wait(smem_u32(&a_full[ar.idx]), ar.ph) & mbar_try_wait(smem_u32(&a_full[a2.idx]), a2.ph);
        return __all_sync(0xffffffffu, both) != 0;
      };
      auto issue = [&]() {
        tc_fence_after();
        const uint32_t a_col = a_col0 + (uint32_t)(ar.idx * kACols);
        const uint64_t bd = bd0 + (uint64_t)(xr.idx * xstep);
        if (elect_one()) {
          mma_f16_tmem_a(d, a_col + 0, bd + 0, idesc, accum);
          mma_f16_tmem_a(d, a_col + 8, bd + 2, idesc, 1u);
          mma_f16_tmem_a(d, a_col + 16, bd + 4, idesc, 1u);
          mma_f16_tmem_a(d, a_col + 24, bd + 6, idesc, 1u);
          mma_commit_mc(&done[xr.idx], (uint16_t)((1u << kPair) - 1u));
        }
        __syncwarp();
        accum = 1u;
        xr.step(1, NX);
        ar.step(1, NA);
      };
      for (int kb = kb0; kb < kb1 && ok; ++kb) {
        const int nch = unit_chunks(kb, c.K);
        if (nch == kChunks) {
#pragma unroll
          for (int g = 0; g < kChunks; g += 2) {
            if (ready2()) {
              issue();
              issue();
            } else if (!stage() || !stage()) {
              ok = false;
              break;
            }
          }
        } else {
          for (int g = 0; g < nch; ++g)
            if (!stage()) {
              ok = false;
              break;
            }
        }
      }
      if (ok && elect_one()) mma_commit(&acc_full[b]);
      __syncwarp();
      i += kb1 - kb0;
    }
    // every MMA the issuing lane issued has finished before tensor memory is freed
    if (elect_one()) {
      mma_commit(drain);
      const uint32_t a = smem_u32(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait_sleep(a, 0u, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp < kEpi0 && c.stall) {
    // test hook: no expansion, so the MMA thread's bounded wait expires
  } else if (warp < kEpi0) {
    // ---------------- weight expansion: thread = weight row r of the tile; set h
    // expands the stages q with q % 2 == h (A slot q % NA, activation slot q % NX)
    const int qd = warp & 3, h = (warp - kConv0) >> 2, r = qd * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)c.acol;
    const int64_t t0 = begin / c.nkb;
    int kb = (int)(begin - t0 * c.nkb), ntp_i = (int)(t0 % c.ntp);
    const int64_t row_bytes = c.K / 4;
    // this set's 16-byte chunks g = g0, g0 + 2, ... of row r of unit (ukb, feature-tile pair up); zeros past N or K
    auto load_unit = [&](int ukb, int up, int g0, uint4* dst) {
      const int64_t n = (int64_t)(kPair * up + rho) * kBM + r;
      const int nch = unit_chunks(ukb, c.K);
      const uint4* src = reinterpret_cast<const uint4*>(c.Wp + n * row_bytes + (int64_t)ukb * (kKB / 4));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int g = g0 + 2 * j;
        dst[j] = (n < c.N && g < nch) ? __ldg(src + g) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    int64_t q0 = 0;  // sequence number of the unit's first stage
    // ring positions of this set's next stage q (q, q + 2, ...: NX and NA are even):
    // its activation slot, the done barrier of stage q - NA, its A slot
    RingPos xp{h, 0u}, dp{h, 0u}, ap{h, 0u};
    uint4 cur[4], nxt[4];
    load_unit(kb, ntp_i, h, cur);
    bool ok = true;
    for (int64_t i = begin; i < end && ok; ++i) {
      const int nch = unit_chunks(kb, c.K);
      const int g0 = (int)((h - q0) & 1);  // this set's first chunk of the unit
      int kb2 = kb + 1, np2 = ntp_i;
      if (kb2 == c.nkb) {
        kb2 = 0;
        if (++np2 == c.ntp) np2 = 0;
      }
      if (i + 1 < end) load_unit(kb2, np2, (int)((h - (q0 + nch)) & 1), nxt);  // one unit ahead
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int g = g0 + 2 * j;
        if (g >= nch) break;
        const int64_t q = q0 + g;
        uint32_t o[32];
        unpack16_f16(cur[j].x, o + 0);
        unpack16_f16(cur[j].y, o + 8);
        unpack16_f16(cur[j].z, o + 16);
        unpack16_f16(cur[j].w, o + 24);
        // the stage's activations have landed (so a_full implies it for the MMA thread) ...
        if (!wait_flag(&x_full[xp.idx], xp.ph, c.err, abort_flag)) {
          ok = false;
          break;
        }
        // ... and the MMAs of stage q - NA, which read this A slot, are done
        if (q >= NA) {
          if (!wait_flag(&done[dp.idx], dp.ph, c.err, abort_flag)) {
            ok = false;
            break;
          }
          dp.step(2, NX);
        }
        tmem_st32(lane_base + (uint32_t)(ap.idx * kACols), o);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[ap.idx]);
        xp.step(2, NX);
        ap.step(2, NA);
      }
      q0 += nch;
      kb = kb2;
      ntp_i = np2;
#pragma unroll
      for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
    }
  } else {
    // ---------------- epilogue: thread = output feature row r of the tile; the
    // two warps of a lane quarter take alternate 16-token chunks
    const int q = warp & 3, eh = (warp - kEpi0) >> 2, r = q * 32 + lane, et = threadIdx.x - 32 * kEpi0;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    pdl_wait();
    const float gamma = __ldg(c.gamma);
    const int first_pt = (int)(begin / c.nkb);  // first feature-tile pair (with its token tile) of the range
    const int me = kPair * cl + rho;            // this CTA's index among the ranks rho
    int lt = 0;
    for (int64_t i = begin; i < end; ++lt) {
      const int64_t pt = i / c.nkb;
      const int kb0 = (int)(i - pt * c.nkb);
      const int kb1 = (int)min((int64_t)c.nkb, kb0 + (end - i));
      i += kb1 - kb0;
      const int b = lt & 1;
      const int64_t mt = pt / c.ntp;
      const int n0 = (kPair * (int)(pt - mt * c.ntp) + rho) * kBM, m0 = (int)(mt * BN);
      float* ts = tscale + b * BN;
      for (int j = et; j < BN; j += 32 * kEpiWarps) {
        const int m = m0 + j;
        ts[j] = m < c.M ? __fdiv_rn(gamma, __ldg(c.s + m)) : 0.0f;
      }
      const bool got = wait_flag(&acc_full[b], (uint32_t)(lt >> 1) & 1u, c.err, abort_flag);
      if (epi_bar_or(!got)) break;  // the scales above are visible, and every warp agrees
      tc_fence_after();
      const int n = n0 + r;
      const uint32_t dcol = lane_base + (uint32_t)(b * c.acc_stride);
      const bool whole = kb0 == 0 && kb1 == c.nkb;
      bool last = whole;
      const int my_slot = 2 * me + ((int)pt == first_pt ? 0 : 1);
      if (!whole) {
        // This CTA is the last contributor if every other k-block of the tile
        // is already counted: it then needs no partial slot of its own.
        // Otherwise it stores its partial sums, then counts its k-blocks (and
        // may still turn out last).
        const int clo = cluster_of(pt * c.nkb, U, c.C);
        uint32_t* counter = c.cnt + kPair * clo + rho;
        const uint32_t mine = (uint32_t)(kb1 - kb0);
        if (et == 0) *last_flag = atomicAdd(counter, 0u) + mine == (uint32_t)c.nkb ? 1u : 0u;
        epi_bar();
        last = *last_flag != 0u;
        if (last) {
          __threadfence();  // the others' partial sums, counted before, are visible
        } else {
          float* slot = c.part + (size_t)my_slot * (BN * kBM);
          for (int j0 = 16 * eh; j0 < BN; j0 += 32) {
            uint32_t v[16];
            tmem_ld16(dcol + (uint32_t)j0, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) slot[(j0 + jj) * kBM + r] = __uint_as_float(v[jj]);
          }
          __threadfence();
          epi_bar();
          if (et == 0) *last_flag = atomicAdd(counter, mine) + mine == (uint32_t)c.nkb ? 1u : 0u;
          epi_bar();
          last = *last_flag != 0u;
          if (last) __threadfence();
        }
      }
      if (last) {
        const int clo = whole ? 0 : cluster_of(pt * c.nkb, U, c.C);
        const int chi = whole ? -1 : cluster_of((pt + 1) * c.nkb - 1, U, c.C);
        // the other contributors' slots; the first is read one chunk ahead (its
        // loads in flight while the current chunk is summed and stored), any
        // further ones in turn
        const float* peer0 = nullptr;
        int npeer = 0;
        for (int cc = clo; cc <= chi; ++cc) {
          if (cc == cl) continue;
          const int cfirst = (int)(((int64_t)cc * U / c.C) / c.nkb);  // first pair of cluster cc
          if (npeer == 0)
            peer0 = c.part + (size_t)(2 * (kPair * cc + rho) + (cfirst == (int)pt ? 0 : 1)) * (BN * kBM);
          ++npeer;
        }
        float p0[16];
        auto fetch = [&](int j0, float (&q0)[16]) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) q0[jj] = npeer > 0 ? __ldcg(peer0 + (j0 + jj) * kBM + r) : 0.0f;
        };
        if (16 * eh < BN) fetch(16 * eh, p0);
        for (int j0 = 16 * eh; j0 < BN; j0 += 32) {
          float n0[16];
          if (j0 + 32 < BN) fetch(j0 + 32, n0);
          uint32_t v[16];
          tmem_ld16(dcol + (uint32_t)j0, v);
          float a[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) a[jj] = __fadd_rn(__uint_as_float(v[jj]), p0[jj]);
          if (npeer > 1) {  // a tile spread over more than two clusters: the rest in turn
            int k = 0;
            for (int cc = clo; cc <= chi; ++cc) {
              if (cc == cl || k++ < 1) continue;
              const int cfirst = (int)(((int64_t)cc * U / c.C) / c.nkb);
              const float* slot =
                  c.part + (size_t)(2 * (kPair * cc + rho) + (cfirst == (int)pt ? 0 : 1)) * (BN * kBM);
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) a[jj] = __fadd_rn(a[jj], __ldcg(slot + (j0 + jj) * kBM + r));
            }
          }
          if (n < c.N) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int m = m0 + j0 + jj;
              if (m < c.M) {
                const int64_t o = (int64_t)m * c.N + n;
                c.y[o] = out_act(__fmul_rn(a[jj], ts[j0 + jj]), c.relu2);
                if (c.acc) c.acc[o] = __float2int_rn(a[jj]);
              }
            }
          }
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) p0[jj] = n0[jj];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }
  __syncthreads();
  // neither CTA leaves while the other may still multicast into it or commit to its barriers
  cluster_sync_all();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The fp16 operand from x_q (one thread per 16-k group; positions p = 4 i + j
// hold k = 4 j + i); block 0 also zeroes the arrival counters.
__global__ void __launch_bounds__(256) x16_sk_prepass_kernel(const uint4* __restrict__ xq, uint64_t ngroups,
                                                             uint4* __restrict__ x16, uint32_t* __restrict__ cnt,
                                                             int ncnt) {
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0u;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < ngroups; i += stride) {
    uint32_t f[8];
    convert_x16_f16(__ldg(xq + i), f);
    x16[2 * i] = make_uint4(f[0], f[1], f[2], f[3]);
    x16[2 * i + 1] = make_uint4(f[4], f[5], f[6], f[7]);
  }
}

struct SkLayout {
  uint8_t* x16;
  float* part;
  uint32_t* cnt;
};

SkLayout sk_layout(void* ws, int64_t M, int64_t K, int num_sms) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  SkLayout l;
  l.x16 = p;
  p += ((size_t)M * (size_t)K * 2 + 255) / 256 * 256;
  l.part = reinterpret_cast<float*>(p);
  p += (size_t)2 * num_sms * gemm_sk_token_tile(M) * kBM * sizeof(float);
  l.cnt = reinterpret_cast<uint32_t*>(p);
  return l;
}

}  // namespace

int gemm_sk_token_tile(int64_t M) {
  const int64_t ntm = (M + kSkMaxTile - 1) / kSkMaxTile;  // token tiles of at most kSkMaxTile
  return (int)(((M + ntm - 1) / ntm + 15) / 16 * 16);
}

size_t gemm_sk_workspace_bytes(int64_t M, int64_t K, int num_sms) {
  return ((size_t)M * (size_t)K * 2 + 255) / 256 * 256 +
         (size_t)2 * num_sms * gemm_sk_token_tile(M) * kBM * sizeof(float) +
         ((size_t)num_sms * sizeof(uint32_t) + 255) / 256 * 256;
}

uint32_t* sk_counters(void* ws, int64_t M, int64_t K, int num_sms) { return sk_layout(ws, M, K, num_sms).cnt; }

cudaError_t launch_x16_sk_prepass(const int8_t* xq, int64_t M, int64_t K, void* ws, int num_sms,
                                  cudaStream_t stream) {
  const SkLayout l = sk_layout(ws, M, K, num_sms);
  const uint64_t ngroups = (uint64_t)M * (uint64_t)K / 16;
  const uint64_t want = (ngroups + 255) / 256;
  const int grid = (int)(want < (uint64_t)num_sms * 8 ? (want ? want : 1) : (uint64_t)num_sms * 8);
  x16_sk_prepass_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(xq), ngroups,
                                                  reinterpret_cast<uint4*>(l.x16), l.cnt, num_sms);
  return cudaGetLastError();
}

namespace {

// Clusters of kPair CTAs that can be resident at once with this much shared
// memory (at most num_sms / kPair), cached per shared-memory size.
int resident_pairs(size_t smem, int num_sms) {
  static std::mutex mu;
  static size_t key_smem[16];
  static int key_sms[16], val[16];
  static int n = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (key_smem[i] == smem && key_sms[i] == num_sms) return val[i];
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_sms / kPair * kPair));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, gemm_f16_sk_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    nclusters = 0;
  }
  if (nclusters > num_sms / kPair) nclusters = num_sms / kPair;
  std::lock_guard<std::mutex> lock(mu);
  if (n < 16) {
    key_smem[n] = smem;
    key_sms[n] = num_sms;
    val[n] = nclusters;
    ++n;
  }
  return nclusters;
}

}  // namespace

cudaError_t launch_gemm_f16_sk(const ForwardArgs& a, void* ws, int num_sms, cudaStream_t stream) {
  const SkLayout l = sk_layout(ws, a.M, a.K, num_sms);
  const int BN = gemm_sk_token_tile(a.M);
  CUtensorMap tx;
  if (!encode_f16_2d_sw128(&tx, l.x16, (uint64_t)a.K, (uint64_t)a.M, (uint32_t)BN)) return cudaErrorInvalidValue;
  const int ntn = (int)((a.N + kBM - 1) / kBM);
  const int ntp = (ntn + kPair - 1) / kPair;
  const int64_t ntm = (a.M + BN - 1) / BN;
  const int nkb = (int)((a.K + kKB - 1) / kKB);
  const int64_t units = (int64_t)ntp * ntm * nkb;
  // tensor memory: two accumulators of BN columns at a 32-column stride, then
  // the expanded-weight slots of 32 columns
  const int acc_stride = (BN + 31) / 32 * 32;
  const int acol = 2 * acc_stride;
  int NA = (512 - acol) / kACols;
  if (NA > kMaxASlots) NA = kMaxASlots;
  if (NA < 2) return cudaErrorInvalidValue;
  // shared memory: the activation ring, a multiple of the producer count
  const size_t xstage = (size_t)BN * kRowB;
  const size_t fixed = 1024 + (2 * kMaxXStages + kMaxASlots + 5) * 8 + 16 + (size_t)2 * BN * 4;
  int NX = (int)((kSmemBudget - fixed) / xstage);
  if (NX > kMaxXStages) NX = kMaxXStages;
  NX -= NX % kXProducers;  // each producer owns the slots = its index mod kXProducers
  if (NX < kXProducers) return cudaErrorInvalidValue;
  // an expanding set reuses an A slot after the stage NA back is done: NA < NX
  // keeps every phase it waits for ahead of the barrier's next one
  if (NA >= NX) NA = NX - 2;
  if (NA < 2) return cudaErrorInvalidValue;
  size_t smem = fixed + (size_t)NX * xstage;
  if (smem < kSmemFloor) smem = kSmemFloor;
  cudaError_t e = cudaFuncSetAttribute(gemm_f16_sk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int C = resident_pairs(smem, num_sms);
  if (C < 1) return cudaErrorInvalidConfiguration;
  if ((int64_t)C > units) C = (int)units;
  SkCfg c{a.Wp, a.gamma, a.s, a.y, a.acc, a.err, l.part, l.cnt, (int)a.M, (int)a.N, (int)a.K, BN, NX, NA,
          acc_stride, acol, ntn, ntp, nkb, C, units, a.relu2 ? 1 : 0, a.test_stall ? 1 : 0};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(kPair * C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // a programmatic dependent of the preceding kernel (the quantisation or the
  // prepass): barrier set-up, tensor-memory allocation and the weight
  // expansion start before it ends; the activation producers and the
  // epilogue wait for it (griddepcontrol.wait) before reading what it wrote
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_f16_sk_kernel, tx, c);
}

}  // namespace bl
