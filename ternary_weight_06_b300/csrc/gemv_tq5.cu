// gemv_tq5.cu -- the BitLinear forward for a few tokens from base-3 packed
// weights, five per byte (1.6 bits per weight: the pages put a ternary
// weight's information at log2(3) = 1.58 bits and the 2B model's weights
// under 2 bits each; yousumm.com transcript, the GPU-plumbing paragraph, and
// anthology note-168 on arXiv 2402.17764, "What it does").
//
// Byte j of a row holds sum_i (q[5j+i] + 1) * 3^i; rows are `pitch` bytes
// (ceil(K/5) rounded up to 16), padded with zero codes.
//
// One CTA per SM.  A producer warp streams the CTA's rows through a ring of
// shared-memory stages with 1-D bulk copies (as the 2-bit GEMV does); 16
// consumer warps split each row's 32-bit words into K slices.  A word holds
// four bytes = 20 weights and meets 20 contiguous activations, which the
// lane keeps in registers as four 4-element groups plus one word of the
// fifth elements.  Decoding is one table lookup per byte: the table maps a
// byte to its codes 0..3 (one word) and code 4 (one byte), and every lane has
// its own copy in its own bank pair (256 entries x 32 lanes x 8 bytes), so
// the lookups of a warp never conflict.  Per word and token that is five
// dp4a; the product is exact in int32, and y = fp32(acc) * fp32(gamma / s)
// as in every other path.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace bl {
namespace {

constexpr int kT5ConsumerWarps = 16;
constexpr int kT5Threads = 32 * (kT5ConsumerWarps + 1);
constexpr int kT5Stages = 3;
constexpr int kT5StageBytesTarget = 32768;
constexpr int kT5LutBytes = 256 * 32 * 8;  // per-lane copies of the 256-entry decode table
constexpr int kT5MaxI = 4;                 // 32-bit weight words per lane and row

struct Tq5Cfg {
  const uint8_t* Wt;
  const float* gamma;
  const int8_t* xq;
  const float* s;
  float* y;
  int32_t* acc;
  uint32_t* err;
  int64_t N, K;
  int pitch, words;  // bytes and 32-bit words per row
  int rows_per_cta, rows_per_stage, nslots;
  int kw, words_per_warp;  // K slices per row and the words of each
  int tok0, ntok;
  int relu2;
  int stall;  // test hook: the producer issues nothing
};

__device__ __forceinline__ bool t5_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code,
                                        volatile uint32_t* abort_flag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(a, parity, kWaitHintNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, code);
      *abort_flag = 1u;
      return false;
    }
  }
}

__device__ __forceinline__ void t5_consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kT5ConsumerWarps) : "memory");
}

// low bytes of a, b, c, d -> bytes 0..3 of one word
__device__ __forceinline__ uint32_t t5_pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

// The 20 activations x[20d .. 20d+19] of word d, as five natural words X0..X4,
// regrouped to match the five-weight bytes: group g (weights 20d + 5g ..
// 20d + 5g + 3) and the fifth elements 20d + 5g + 4 of the four groups.
__device__ __forceinline__ void t5_regroup(uint32_t X0, uint32_t X1, uint32_t X2, uint32_t X3, uint32_t X4,
                                           uint32_t (&ga)[4], uint32_t& gb) {
  ga[0] = X0;                           // x0 x1 x2 x3
  ga[1] = __byte_perm(X1, X2, 0x4321);  // x5 x6 x7 x8
  ga[2] = __byte_perm(X2, X3, 0x5432);  // x10 x11 x12 x13
  ga[3] = __byte_perm(X3, X4, 0x6543);  // x15 x16 x17 x18
  gb = __byte_perm(__byte_perm(X1, X2, 0x0050u), __byte_perm(X3, X4, 0x0072u), 0x5410u);  // x4 x9 x14 x19
}

template <int MT, int I>
__global__ void __launch_bounds__(kT5Threads, 1) gemv_tq5_kernel(const Tq5Cfg c) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint2* lut = reinterpret_cast<uint2*>(smem);  // [256][32]: entry b, copy of lane l at b * 32 + l
  uint8_t* ring = smem + kT5LutBytes;
  const int SR = c.rows_per_stage, NS = c.nslots;
  const int stage_bytes = SR * c.pitch;  // multiple of 16
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + NS * stage_bytes);
  uint64_t* empty = full + kT5Stages;
  int32_t* acc_sm = reinterpret_cast<int32_t*>(empty + kT5Stages);  // [rows_per_cta][MT]
  float* tsc_sm = reinterpret_cast<float*>(acc_sm + c.rows_per_cta * MT);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(tsc_sm + MT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = (int64_t)blockIdx.x * c.rows_per_cta;
  const int nrows = (int)min((int64_t)c.rows_per_cta, c.N - row0);
  const int nstages = (nrows + SR - 1) / SR;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kT5Stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kT5ConsumerWarps);
    }
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  for (int i = threadIdx.x; i < c.rows_per_cta * MT; i += blockDim.x) acc_sm[i] = 0;
  __syncthreads();

  if (warp == kT5ConsumerWarps) {
    // ---------------- producer: the CTA's rows, stage by stage
    if (lane == 0) {
      int issued = 0;
      for (int st = 0; st < (c.stall ? 0 : nstages); ++st) {
        const int slot = st % NS;
        if (st >= NS &&
            !t5_wait(&empty[slot], (uint32_t)((st / NS) - 1) & 1u, c.err, kErrGemvEmptyWait, abort_flag))
          break;
        const int rows = min(SR, nrows - st * SR);
        const uint32_t bytes = (uint32_t)(rows * c.pitch);
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(ring + slot * stage_bytes, c.Wt + (row0 + (int64_t)st * SR) * c.pitch, bytes, &full[slot]);
        issued = st + 1;
      }
      if (*abort_flag) {
        // let every copy this CTA started land before its shared memory goes away
        for (int st = (issued > NS ? issued - NS : 0); st < issued; ++st) {
          const uint32_t a = smem_u32(&full[st % NS]), par = (uint32_t)(st / NS) & 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait_sleep(a, par, kWaitHintNs) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    return;
  }

  // ---------------- consumers
  // decode table (while the first stages stream in): entry b holds the codes
  // d_i - 1 of its base-3 digits 0..3 in bytes 0..3 of .x and of digit 4 in
  // byte 0 of .y; bytes above 242 (never written) decode to zero codes
  for (int e = threadIdx.x; e < 256 * 32; e += 32 * kT5ConsumerWarps) {
    const int b = e >> 5;
    uint32_t lo = 0u, hi = 0u;
    if (b < 243) {
      int v = b;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        lo |= (uint32_t)(uint8_t)(int8_t)(v % 3 - 1) << (8 * i);
        v /= 3;
      }
      hi = (uint32_t)(uint8_t)(int8_t)(v - 1);
    }
    lut[e] = make_uint2(lo, hi);
  }
  if (threadIdx.x < MT) {
    const int t = threadIdx.x;
    tsc_sm[t] = t < c.ntok ? __fdiv_rn(__ldg(c.gamma), __ldg(c.s + c.tok0 + t)) : 0.0f;
  }

  const int kwi = warp % c.kw, rg = warp / c.kw, nrg = kT5ConsumerWarps / c.kw;
  const int wbeg = kwi * c.words_per_warp;
  const int wend = min(wbeg + c.words_per_warp, c.words);

  // activations of this lane's words, regrouped (zeros past K and past the slice)
  uint32_t xa[I][4][MT], xb[I][MT];
#pragma unroll
  for (int i = 0; i < I; ++i) {
    const int d = wbeg + lane + 32 * i;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      uint32_t X[5] = {0u, 0u, 0u, 0u, 0u};
      if (d < wend && t < c.ntok) {
        const uint32_t* xrow = reinterpret_cast<const uint32_t*>(c.xq + (int64_t)(c.tok0 + t) * c.K);
#pragma unroll
        for (int u = 0; u < 5; ++u) {
          const int64_t w = 5 * (int64_t)d + u;  // activation word: bytes 4w .. 4w + 3
          if (4 * w < c.K) X[u] = __ldg(xrow + w);
        }
      }
      uint32_t ga[4], gb;
      t5_regroup(X[0], X[1], X[2], X[3], X[4], ga, gb);
#pragma unroll
      for (int g = 0; g < 4; ++g) xa[i][g][t] = ga[g];
      xb[i][t] = gb;
    }
  }
  t5_consumer_bar();  // the decode table is complete

  const uint2* lut_lane = lut + lane;
  for (int st = 0; st < nstages; ++st) {
    const int slot = st % NS;
    const int rows = min(SR, nrows - st * SR);
    const bool ok = t5_wait(&full[slot], (uint32_t)(st / NS) & 1u, c.err, kErrGemvFullWait, abort_flag);
    if (ok) {
      const uint8_t* base = ring + slot * stage_bytes;
      for (int r = rg; r < rows; r += nrg) {
        int32_t a[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) a[t] = 0;
        const uint32_t* rw = reinterpret_cast<const uint32_t*>(base + r * c.pitch);
#pragma unroll
        for (int i = 0; i < I; ++i) {
          const int d = wbeg + lane + 32 * i;
          if (d < wend) {
            const uint32_t P = rw[d];
            const uint2 e0 = lut_lane[(P & 0xffu) << 5];
            const uint2 e1 = lut_lane[((P >> 8) & 0xffu) << 5];
            const uint2 e2 = lut_lane[((P >> 16) & 0xffu) << 5];
            const uint2 e3 = lut_lane[(P >> 24) << 5];
            const uint32_t c4 = t5_pack_low_bytes(e0.y, e1.y, e2.y, e3.y);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              int32_t v = __dp4a((int)e0.x, (int)xa[i][0][t], a[t]);
              v = __dp4a((int)e1.x, (int)xa[i][1][t], v);
              v = __dp4a((int)e2.x, (int)xa[i][2][t], v);
              v = __dp4a((int)e3.x, (int)xa[i][3][t], v);
              a[t] = __dp4a((int)c4, (int)xb[i][t], v);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const int32_t v = __reduce_add_sync(0xffffffffu, a[t]);
          if (lane == 0) {
            int32_t* dst = &acc_sm[(st * SR + r) * MT + t];
            if (c.kw == 1) *dst = v;
            else atomicAdd(dst, v);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  t5_consumer_bar();
  if (*abort_flag == 0u) {
    for (int idx = threadIdx.x; idx < nrows * c.ntok; idx += 32 * kT5ConsumerWarps) {
      const int t = idx / nrows, r = idx - t * nrows;
      const int32_t v = acc_sm[r * MT + t];
      const int64_t o = (int64_t)(c.tok0 + t) * c.N + row0 + r;
      c.y[o] = out_act(__fmul_rn(__int2float_rn(v), tsc_sm[t]), c.relu2);
      if (c.acc) c.acc[o] = v;
    }
  }
}

template <int MT, int I>
cudaError_t t5_launch(const Tq5Cfg& c, int grid, size_t smem, cudaStream_t stream) {
  auto kern = gemv_tq5_kernel<MT, I>;
  if (cudaError_t e = set_smem_attrs(kern, smem)) return e;
  kern<<<grid, kT5Threads, smem, stream>>>(c);
  return cudaGetLastError();
}

// words per lane I <= kT5MaxI / MT: at most 20 activation registers (5 per
// word and token), so that 17 warps per CTA run without spills
template <int MT>
cudaError_t t5_dispatch(const Tq5Cfg& c, int I, int grid, size_t smem, cudaStream_t stream) {
  if constexpr (MT == 4) {
    return I == 1 ? t5_launch<MT, 1>(c, grid, smem, stream) : cudaErrorInvalidValue;
  } else if constexpr (MT == 2) {
    switch (I) {
      case 1: return t5_launch<MT, 1>(c, grid, smem, stream);
      case 2: return t5_launch<MT, 2>(c, grid, smem, stream);
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (I) {
      case 1: return t5_launch<MT, 1>(c, grid, smem, stream);
      case 2: return t5_launch<MT, 2>(c, grid, smem, stream);
      case 3: return t5_launch<MT, 3>(c, grid, smem, stream);
      case 4: return t5_launch<MT, 4>(c, grid, smem, stream);
      default: return cudaErrorInvalidValue;
    }
  }
}

}  // namespace

cudaError_t launch_gemv_tq5(const ForwardArgs& a, int64_t pitch, int num_sms, cudaStream_t stream) {
  Tq5Cfg c{};
  c.Wt = a.Wp;
  c.gamma = a.gamma;
  c.xq = a.xq;
  c.s = a.s;
  c.y = a.y;
  c.acc = a.acc;
  c.err = a.err;
  c.N = a.N;
  c.K = a.K;
  c.pitch = (int)pitch;
  c.words = (int)(pitch / 4);
  c.relu2 = a.relu2 ? 1 : 0;
  c.stall = a.test_stall ? 1 : 0;

  int grid = (int)(a.N < num_sms ? a.N : num_sms);
  c.rows_per_cta = (int)((a.N + grid - 1) / grid);
  grid = (int)((a.N + c.rows_per_cta - 1) / c.rows_per_cta);
  int sr = kT5StageBytesTarget / c.pitch;
  if (sr < 1) sr = 1;
  if (sr > c.rows_per_cta) sr = c.rows_per_cta;
  c.rows_per_stage = sr;
  const int max_stages = (c.rows_per_cta + sr - 1) / sr;
  c.nslots = max_stages < kT5Stages ? max_stages : kT5Stages;

  // tokens per pass (4, 2 or 1) and K slices per row: the fewest slices whose
  // words per lane fit the activation registers of that many tokens
  int mt = a.M >= 4 ? 4 : a.M >= 2 ? 2 : 1, kw = 0, I = 0;
  for (; mt >= 1 && kw == 0; mt /= 2) {
    for (int k = 1; k <= kT5ConsumerWarps; k *= 2) {
      const int wpw = (c.words + k - 1) / k;
      const int i = (wpw + 31) / 32;
      if (i <= kT5MaxI / mt) {
        kw = k;
        I = i;
        break;
      }
    }
    if (kw) break;
  }
  if (kw == 0) return cudaErrorInvalidValue;  // K beyond the kernel's register budget
  c.kw = kw;
  c.words_per_warp = (c.words + kw - 1) / kw;
  const size_t smem = (size_t)kT5LutBytes + (size_t)c.nslots * sr * c.pitch + 2 * kT5Stages * sizeof(uint64_t) +
                      (size_t)c.rows_per_cta * mt * sizeof(int32_t) + mt * sizeof(float) + 16;

  for (int64_t t0 = 0; t0 < a.M; t0 += mt) {
    c.tok0 = (int)t0;
    c.ntok = (int)(a.M - t0 < mt ? a.M - t0 : mt);
    cudaError_t e = mt == 4   ? t5_dispatch<4>(c, I, grid, smem, stream)
                    : mt == 2 ? t5_dispatch<2>(c, I, grid, smem, stream)
                              : t5_dispatch<1>(c, I, grid, smem, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace bl
