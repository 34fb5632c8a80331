// gemv.cu -- streaming ternary GEMV for a few tokens (decode), with the
// dequant epilogue fused.
//
// The work is bounded by reading the packed weights from HBM once ("bundles
// four chips into a single byte, slides that bundle across the GPU highway,
// unpacks it right next to the math engine": yousumm.com BitNet b1.58 2B4T
// transcript; memory and bandwidth savings are the measured part: anthology
// note-168, "The part that is a bet rather than a measurement").
//
// Layout of the work:
//   * one CTA per SM, each owning a contiguous block of ~N/#SM output rows;
//     because packed rows are contiguous, that block is one contiguous byte
//     range, streamed through a ring of shared-memory stages by 1-D bulk
//     async copies (one elected producer thread, mbarrier completion);
//   * consumer warps own a fixed slice of K: lane l of k-warp kw handles the
//     16-code words w = kw*Cw + l + 32 j of every row.  Their activations are
//     loaded once into registers, so shared memory carries weights only;
//   * unpacking a 32-bit word P of 16 codes takes two ops per 4 weights:
//     S_i = (P >> 2i) & 0x03030303 holds the codes of weights 4j+i (j = 0..3)
//     as bytes in {0,1,2}.  The matching activation word X'_i holds x[4j+i]
//     (a 4x4 byte transpose of the natural 16 activations, done once), so
//       sum_k (c_k - 1) x_k = sum_i dp4a(S_i, X'_i) - sum_k x_k,
//     an exact int32 sum ("only involves integer addition");
//   * y[m,n] = fp32(acc) * fp32(gamma / s[m]) is written straight from the
//     reduced accumulator (and acc itself when requested).
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace bl {
namespace {

constexpr int kStages = 6;
constexpr int kStageBytesTarget = 16384;
constexpr int kMaxRowsPerStage = 128;
constexpr int kMaxConsumerWarps = 16;

struct GemvCfg {
  const uint8_t* Wp;
  const float* gamma;
  const int8_t* xq;
  const float* s;
  float* y;
  int32_t* acc;
  uint32_t* err;
  int64_t N, K;
  int tok0, ntok;  // tokens of this launch
  int rows_per_cta, rows_per_stage, row_bytes;
  int kw, rwp, words_per_row, words_per_warp, J;
};

__device__ __forceinline__ void transpose4x4(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, uint32_t* o) {
  const uint32_t t0 = __byte_perm(x0, x1, 0x5140), t1 = __byte_perm(x2, x3, 0x5140);
  const uint32_t t2 = __byte_perm(x0, x1, 0x7362), t3 = __byte_perm(x2, x3, 0x7362);
  o[0] = __byte_perm(t0, t1, 0x5410);
  o[1] = __byte_perm(t0, t1, 0x7632);
  o[2] = __byte_perm(t2, t3, 0x5410);
  o[3] = __byte_perm(t2, t3, 0x7632);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code,
                                              volatile uint32_t* abort_flag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, code);
      *abort_flag = 1u;
      return false;
    }
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int MT, int JMAX>
__global__ void __launch_bounds__(32 * (1 + kMaxConsumerWarps)) gemv_kernel(const GemvCfg c) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int SR = c.rows_per_stage;
  const int stage_bytes = SR * c.row_bytes;  // multiple of 16
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage_bytes);
  uint64_t* empty = full + kStages;
  int32_t* red = reinterpret_cast<int32_t*>(empty + kStages);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(red + kStages * SR * MT);
  const int n_consumers = c.kw * c.rwp;

  const int64_t row0 = (int64_t)blockIdx.x * c.rows_per_cta;
  const int64_t row_end = min(row0 + (int64_t)c.rows_per_cta, c.N);
  const int nrows = (int)(row_end - row0);
  const int nstages = (nrows + SR - 1) / SR;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], (uint32_t)n_consumers);
    }
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  for (int i = threadIdx.x; i < kStages * SR * MT; i += blockDim.x) red[i] = 0;
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer: one elected thread streams the row block.
    if (lane == 0) {
      int issued = 0;
      for (int st = 0; st < nstages; ++st) {
        const int slot = st % kStages;
        if (st >= kStages &&
            !wait_or_abort(&empty[slot], (uint32_t)((st / kStages) - 1) & 1u, c.err, kErrGemvEmptyWait, abort_flag))
          break;
        const int rows = min(SR, nrows - st * SR);
        const uint32_t bytes = (uint32_t)(rows * c.row_bytes);
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(smem + slot * stage_bytes, c.Wp + (row0 + (int64_t)st * SR) * c.row_bytes, bytes, &full[slot]);
        issued = st + 1;
      }
      if (*abort_flag) {
        // Let every copy this CTA started land before its shared memory goes away.
        for (int st = (issued > kStages ? issued - kStages : 0); st < issued; ++st) {
          uint64_t* bar = &full[st % kStages];
          const uint32_t a = smem_u32(bar), par = (uint32_t)(st / kStages) & 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, par) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    return;
  }

  // ---------------- consumers
  const int cw = warp - 1;
  const int kw = cw % c.kw, rw = cw / c.kw;
  pdl_wait();  // activations and scales may come from the preceding kernel

  const int wbeg = kw * c.words_per_warp;
  const int wend = min(wbeg + c.words_per_warp, c.words_per_row);
  uint32_t xr[JMAX][4][MT];
  int32_t xsum[MT];
  float tscale[MT];
  const float gamma = __ldg(c.gamma);
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    xsum[t] = 0;
    tscale[t] = t < c.ntok ? __fdiv_rn(gamma, __ldg(c.s + c.tok0 + t)) : 0.0f;
  }
#pragma unroll
  for (int j = 0; j < JMAX; ++j) {
    const int w = wbeg + lane + 32 * j;
    const bool valid = j < c.J && w < wend;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      if (valid && t < c.ntok) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(c.xq + (int64_t)(c.tok0 + t) * c.K) + w);
        uint32_t o[4];
        transpose4x4((uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w, o);
#pragma unroll
        for (int i = 0; i < 4; ++i) xr[j][i][t] = o[i];
        xsum[t] = __dp4a(v.x, 0x01010101, __dp4a(v.y, 0x01010101, __dp4a(v.z, 0x01010101, __dp4a(v.w, 0x01010101, xsum[t]))));
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) xr[j][i][t] = 0u;
      }
    }
  }

  for (int st = 0; st < nstages; ++st) {
    const int slot = st % kStages;
    const int rows = min(SR, nrows - st * SR);
    const bool ok = wait_or_abort(&full[slot], (uint32_t)(st / kStages) & 1u, c.err, kErrGemvFullWait, abort_flag);
    if (ok) {
      const uint8_t* base = smem + slot * stage_bytes;
      for (int r = rw; r < rows; r += c.rwp) {
        const uint32_t* rowp = reinterpret_cast<const uint32_t*>(base + r * c.row_bytes);
        int32_t a[MT][4];
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) a[t][i] = 0;
#pragma unroll
        for (int j = 0; j < JMAX; ++j) {
          const int w = wbeg + lane + 32 * j;
          if (j < c.J && w < wend) {
            const uint32_t P = rowp[w];
            const uint32_t S[4] = {P & 0x03030303u, (P >> 2) & 0x03030303u, (P >> 4) & 0x03030303u,
                                   (P >> 6) & 0x03030303u};
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
              for (int i = 0; i < 4; ++i) a[t][i] = __dp4a((int)S[i], (int)xr[j][i][t], a[t][i]);
          }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          int32_t v = a[t][0] + a[t][1] + a[t][2] + a[t][3] - xsum[t];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane == 0 && t < c.ntok) {
            if (c.kw == 1) {
              const int64_t n = row0 + (int64_t)st * SR + r;
              const int64_t o = (int64_t)(c.tok0 + t) * c.N + n;
              c.y[o] = __fmul_rn(__int2float_rn(v), tscale[t]);
              if (c.acc) c.acc[o] = v;
            } else {
              atomicAdd(&red[(slot * SR + r) * MT + t], v);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (c.kw > 1) {
      named_bar_sync(1, n_consumers * 32);
      if (ok) {
        for (int idx = cw * 32 + lane; idx < rows * MT; idx += n_consumers * 32) {
          const int r = idx / MT, t = idx % MT;
          int32_t* cell = &red[(slot * SR + r) * MT + t];
          if (t < c.ntok) {
            const int32_t v = *cell;
            const int64_t n = row0 + (int64_t)st * SR + r;
            const int64_t o = (int64_t)(c.tok0 + t) * c.N + n;
            float ts = tscale[0];
#pragma unroll
            for (int u = 1; u < MT; ++u)
              if (t == u) ts = tscale[u];
            c.y[o] = __fmul_rn(__int2float_rn(v), ts);
            if (c.acc) c.acc[o] = v;
          }
          *cell = 0;
        }
      }
    }
  }
}

template <int MT, int JMAX>
cudaError_t launch_one(const GemvCfg& c, int grid, cudaStream_t stream) {
  const int threads = 32 * (1 + c.kw * c.rwp);
  const size_t smem = (size_t)kStages * c.rows_per_stage * c.row_bytes + 2 * kStages * sizeof(uint64_t) +
                      (size_t)kStages * c.rows_per_stage * MT * sizeof(int32_t) + 16;
  auto kern = gemv_kernel<MT, JMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, threads, smem, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const ForwardArgs& a, int num_sms, cudaStream_t stream) {
  GemvCfg c{};
  c.Wp = a.Wp;
  c.gamma = a.gamma;
  c.xq = a.xq;
  c.s = a.s;
  c.y = a.y;
  c.acc = a.acc;
  c.err = a.err;
  c.N = a.N;
  c.K = a.K;
  c.row_bytes = (int)(a.K / 4);
  c.words_per_row = (int)(a.K / 16);

  int grid = (int)(a.N < num_sms ? a.N : num_sms);
  c.rows_per_cta = (int)((a.N + grid - 1) / grid);
  grid = (int)((a.N + c.rows_per_cta - 1) / c.rows_per_cta);
  int sr = kStageBytesTarget / c.row_bytes;
  if (sr > kMaxRowsPerStage) sr = kMaxRowsPerStage;
  if (sr < 1) sr = 1;
  if (sr > c.rows_per_cta) sr = c.rows_per_cta;
  c.rows_per_stage = sr;

  // tokens per pass: the largest of 4, 2, 1 (<= M) whose k-split fits 16 warps.
  // Each lane keeps 64 activation registers: JMAX words x 4 x MT tokens.
  auto kw_for = [&](int jmax) { return (c.words_per_row + 32 * jmax - 1) / (32 * jmax); };
  int mt = 1;
  if (a.M >= 4 && kw_for(4) <= kMaxConsumerWarps) mt = 4;
  else if (a.M >= 2 && kw_for(8) <= kMaxConsumerWarps) mt = 2;
  const int jmax = 16 / mt;
  c.kw = kw_for(jmax);
  if (c.kw > kMaxConsumerWarps) return cudaErrorNotSupported;
  c.words_per_warp = (c.words_per_row + c.kw - 1) / c.kw;
  c.J = (c.words_per_warp + 31) / 32;
  c.rwp = kMaxConsumerWarps / c.kw;
  if (c.rwp < 1) c.rwp = 1;

  for (int64_t t0 = 0; t0 < a.M; t0 += mt) {
    c.tok0 = (int)t0;
    c.ntok = (int)(a.M - t0 < mt ? a.M - t0 : mt);
    cudaError_t e;
    if (mt == 4) e = launch_one<4, 4>(c, grid, stream);
    else if (mt == 2) e = launch_one<2, 8>(c, grid, stream);
    else e = launch_one<1, 16>(c, grid, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace bl
