// gemv.cu -- streaming ternary GEMV for a few tokens (decode), with the
// dequant epilogue fused, and optionally the activation quantisation too.
//
// The work is bounded by reading the packed weights from HBM once: four
// weights travel in each byte and are expanded only where they are multiplied
// (yousumm.com BitNet b1.58 2B4T transcript, the paragraph on running the
// model on graphics cards); the memory and bandwidth savings are what the
// method has measured (anthology note-168, "The part that is a bet rather
// than a measurement").
//
// Layout of the work:
//   * up to two CTAs per SM; each owns a contiguous block of output rows.
//     Packed rows are contiguous, so the block is one byte range, streamed
//     into a ring of shared-memory stages by 1-D bulk async copies issued by
//     one producer thread (mbarrier completion, bounded waits);
//   * the copies are issued BEFORE the kernel waits on its predecessor
//     (griddepcontrol.wait), and the kernel lets its successor launch early
//     (griddepcontrol.launch_dependents).  Under programmatic dependent launch
//     a chain of layers streams the next layer's weights while the previous
//     layer finishes; registers and shared memory leave room for a third CTA
//     per SM for that;
//   * consumer warps own a fixed K slice: lane l of k-warp kw handles the
//     16-code words w = kw*Cw + l + 32 j (j < J, J fixed at compile time) of
//     every row, with the matching activations held in registers;
//   * a 32-bit word P holds 16 codes c in {0,1,2}.  P & (3 << 2i) keeps, in
//     byte j, the code of weight 4j+i scaled by 4^i (at most 128, so it is a
//     valid unsigned byte).  With the activation word X'_i holding x[4j+i]
//     (a 4x4 byte transpose of the natural 16 activations, done once),
//       A_i += dp4a.u32.s32(P & (3 << 2i), X'_i)
//     accumulates 4^i * sum c x over plane i: one AND and one dp4a per four
//     weights and token.  At the end of a row segment
//       sum_k (c_k - 1) x_k = A_0 + A_1/4 + A_2/16 + A_3/64 - sum_k x_k,
//     where each division is an exact arithmetic shift (A_i is a multiple of
//     4^i).  Every step is an exact int32 sum ("only involves integer
//     addition");
//   * each warp reduces its RI x MT row-token sums across lanes with a
//     butterfly that halves the value count per exchange (RI*MT - 1 + 5 -
//     log2(RI*MT) shuffles instead of 5 per value), adds them into a per-CTA
//     shared accumulator, and after the last stage the CTA writes
//     y = fp32(acc) * fp32(gamma / s[m]) with coalesced stores.
// The fused variant quantises X itself (per-token absmax; the same IEEE
// operations as the stand-alone kernel, so x_q and s are bit-identical); the
// first CTA also writes x_q and s out.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace bl {
namespace {

constexpr int kStages = 3;
constexpr int kStageBytesTarget = 32768;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kCtasPerSm = 2;  // CTAs of one launch per SM (a third slot stays free for the next launch)
constexpr float kActClampEps = 1e-5f;

struct GemvCfg {
  const uint8_t* Wp;
  const float* gamma;
  const int8_t* xq_in;  // two-call path: quantised activations
  const float* s_in;    // two-call path: per-token scales
  const void* X;        // fused: raw activations
  int8_t* xq_out;       // fused: x_q output (first CTA writes it)
  float* s_out;         // fused: s output
  float* y;
  int32_t* acc;
  uint32_t* err;
  int64_t N, K;
  int tok0, ntok;  // tokens of this launch (<= MT)
  int x_bf16;
  int rows_per_cta, rows_per_stage, row_bytes, nslots;  // nslots <= kStages ring slots
  int kw, words_per_row, words_per_warp;
  int test_stall;  // test hook: the producer issues no copies, so the bounded waits expire
  int relu2;       // epilogue applies the squared ReLU
};

__device__ __forceinline__ void transpose4x4(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, uint32_t* o) {
  const uint32_t t0 = __byte_perm(x0, x1, 0x5140), t1 = __byte_perm(x2, x3, 0x5140);
  const uint32_t t2 = __byte_perm(x0, x1, 0x7362), t3 = __byte_perm(x2, x3, 0x7362);
  o[0] = __byte_perm(t0, t1, 0x5410);
  o[1] = __byte_perm(t0, t1, 0x7632);
  o[2] = __byte_perm(t2, t3, 0x5410);
  o[3] = __byte_perm(t2, t3, 0x7632);
}

// 4-way dot product of unsigned bytes a with signed bytes b, plus c.
__device__ __forceinline__ int32_t dp4a_us(uint32_t a, uint32_t b, int32_t c) {
  int32_t d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Sum of V values (index v) over the 32 lanes of a warp.  Each exchange step
// s sends half of the remaining values to the partner lane (lane ^ (16 >> s))
// and keeps the other half, so after log2(V) steps each lane holds one partial
// sum; plain xor-steps finish the reduction.  Lane l returns the total of
// value index reduce_index<V>(l).
template <int V>
struct Log2 {
  static constexpr int value = V <= 1 ? 0 : 1 + Log2<V / 2>::value;
};
template <>
struct Log2<1> {
  static constexpr int value = 0;
};

template <int V>
__device__ __forceinline__ int32_t butterfly_sum(int32_t (&v)[V], int lane) {
  constexpr int kSteps = Log2<V>::value;
#pragma unroll
  for (int s = 0; s < kSteps; ++s) {
    const int half = V >> (s + 1);
    const int o = 16 >> s;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const int32_t send = upper ? v[k] : v[k + half];
      const int32_t keep = upper ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  int32_t r = v[0];
#pragma unroll
  for (int o = 16 >> kSteps; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

template <int V>
__device__ __forceinline__ int reduce_index(int lane) {
  constexpr int kSteps = Log2<V>::value;
  int idx = 0;
#pragma unroll
  for (int s = 0; s < kSteps; ++s)
    if (lane & (16 >> s)) idx += V >> (s + 1);
  return idx;
}

// Lanes that write a reduced value: one per value index.
template <int V>
__device__ __forceinline__ bool reduce_writer(int lane) {
  constexpr int kSteps = Log2<V>::value;
  return (lane & ((32 >> kSteps) - 1)) == 0;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code,
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

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory"); }

__device__ __forceinline__ uint32_t q8(float x, float s) {
  int q = __float2int_rn(__fmul_rn(x, s));
  q = min(max(q, -128), 127);
  return (uint32_t)q & 0xffu;
}

// 16 bf16 activations (two 16-byte chunks), quantised, as 4 natural int8 words.
__device__ __forceinline__ void quant16_bf16(uint4 a, uint4 b, float s, uint32_t* out) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    out[i] = q8(__uint_as_float(w[2 * i] << 16), s) | (q8(__uint_as_float(w[2 * i] & 0xffff0000u), s) << 8) |
             (q8(__uint_as_float(w[2 * i + 1] << 16), s) << 16) |
             (q8(__uint_as_float(w[2 * i + 1] & 0xffff0000u), s) << 24);
}

__device__ __forceinline__ uint32_t absmax_bits_bf16(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max((w[i] << 16) & 0x7fff0000u, w[i] & 0x7fff0000u));
  return m;
}

// 16 activations of a token row starting at element k0, quantised, as 4 natural int8 words.
__device__ __forceinline__ void quant16(const void* xrow, int x_bf16, int64_t k0, float s, uint32_t* out) {
  if (x_bf16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xrow) + k0);
    quant16_bf16(__ldg(p), __ldg(p + 1), s, out);
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(xrow) + k0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(p + i);
      out[i] = q8(v.x, s) | (q8(v.y, s) << 8) | (q8(v.z, s) << 16) | (q8(v.w, s) << 24);
    }
  }
}

// RI: rows each warp takes per iteration (its butterfly reduces RI * MT values at once).
template <int MT, int J, int RI, bool FUSED>
__global__ void __launch_bounds__(kThreads, kCtasPerSm + 1) gemv_kernel(const GemvCfg c) {
  constexpr int V = RI * MT;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int SR = c.rows_per_stage;
  const int stage_bytes = SR * c.row_bytes;  // multiple of 16
  const int NS = c.nslots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * stage_bytes);
  uint64_t* empty = full + kStages;
  int32_t* acc_sm = reinterpret_cast<int32_t*>(empty + kStages);                   // [rows_per_cta][MT]
  uint32_t* amax_sm = reinterpret_cast<uint32_t*>(acc_sm + c.rows_per_cta * MT);  // [kConsumerWarps][MT]
  float* tsc_sm = reinterpret_cast<float*>(amax_sm + kConsumerWarps * MT);       // [MT]
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(tsc_sm + MT);

  const int64_t row0 = (int64_t)blockIdx.x * c.rows_per_cta;
  const int nrows = (int)min((int64_t)c.rows_per_cta, c.N - row0);
  const int nstages = (nrows + SR - 1) / SR;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  for (int i = threadIdx.x; i < c.rows_per_cta * MT; i += blockDim.x) acc_sm[i] = 0;
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer: weights only, so it may run ahead of griddepcontrol.wait
    if (lane == 0) {
      int issued = 0;
      for (int st = 0; st < (c.test_stall ? 0 : nstages); ++st) {
        const int slot = st % NS;
        if (st >= NS && !wait_or_abort(&empty[slot], (uint32_t)((st / NS) - 1) & 1u, c.err, kErrGemvEmptyWait,
                                       abort_flag))
          break;
        const int rows = min(SR, nrows - st * SR);
        const uint32_t bytes = (uint32_t)(rows * c.row_bytes);
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(smem + slot * stage_bytes, c.Wp + (row0 + (int64_t)st * SR) * c.row_bytes, bytes, &full[slot]);
        issued = st + 1;
        if (st == min(nstages, NS) - 1) pdl_launch_dependents();
      }
      if (*abort_flag) {
        // Let every copy this CTA started land before its shared memory goes away.
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
  const int kwi = warp % c.kw, rg = warp / c.kw, nrg = kConsumerWarps / c.kw;
  pdl_wait();  // activations, scales and gamma may come from the preceding kernel
  const int wbeg = kwi * c.words_per_warp;
  const int wend = min(wbeg + c.words_per_warp, c.words_per_row);
  const float gamma = __ldg(c.gamma);

  float s_tok[MT];
  // One-pass fused prologue (one token, bf16, at most 4 words per lane): each
  // lane loads only its own words of X, once; the row groups of the CTA cover
  // the row, so the CTA-wide maximum of the lanes' maxima is max|x|; the lane
  // then quantises from the registers it loaded.
  constexpr bool kOnePassShape = FUSED && MT == 1 && J <= 4;
  constexpr int kRawJ = kOnePassShape ? J : 1;
  uint4 raw[kRawJ][2];
  const bool onepass = kOnePassShape && c.x_bf16 && c.ntok == 1;
  if (FUSED && onepass) {
    const uint4* xrow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(c.X) + (int64_t)c.tok0 * c.K);
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < kRawJ; ++j) {
      const int w = wbeg + lane + 32 * j;
      if (w < wend) {
        raw[j][0] = __ldg(xrow + 2 * w);
        raw[j][1] = __ldg(xrow + 2 * w + 1);
      } else {
        raw[j][0] = raw[j][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int j = 0; j < kRawJ; ++j) m = max(m, max(absmax_bits_bf16(raw[j][0]), absmax_bits_bf16(raw[j][1])));
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) amax_sm[warp] = m;
    consumer_bar();
    uint32_t mm = 0;
#pragma unroll
    for (int w8 = 0; w8 < kConsumerWarps; ++w8) mm = max(mm, amax_sm[w8]);
    float a = __uint_as_float(mm);
    if (a < kActClampEps) a = kActClampEps;
    s_tok[0] = __fdiv_rn(127.0f, a);
  } else if (FUSED) {
    // per-token absmax over the whole row: the row is read in 16-byte chunks,
    // kChunksInFlight per thread issued together so a batch costs one round trip
    constexpr int kChunksInFlight = 8;
    constexpr int kCT = 32 * kConsumerWarps;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      uint32_t m = 0;
      if (t < c.ntok) {
        const int64_t esz = c.x_bf16 ? 2 : 4;
        const uint4* row = reinterpret_cast<const uint4*>(static_cast<const char*>(c.X) + (c.tok0 + t) * c.K * esz);
        const int nchunks = (int)(c.K * esz / 16);
        for (int q0 = threadIdx.x; q0 < nchunks; q0 += kCT * kChunksInFlight) {
          uint4 v[kChunksInFlight];
#pragma unroll
          for (int u = 0; u < kChunksInFlight; ++u)
            v[u] = q0 + u * kCT < nchunks ? __ldg(row + q0 + u * kCT) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int u = 0; u < kChunksInFlight; ++u) {
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
              m = c.x_bf16 ? max(m, max((w[i] << 16) & 0x7fff0000u, w[i] & 0x7fff0000u)) : max(m, w[i] & 0x7fffffffu);
          }
        }
      }
      m = __reduce_max_sync(0xffffffffu, m);
      if (lane == 0) amax_sm[warp * MT + t] = m;
    }
    consumer_bar();
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      uint32_t m = 0;
#pragma unroll
      for (int w8 = 0; w8 < kConsumerWarps; ++w8) m = max(m, amax_sm[w8 * MT + t]);
      float a = __uint_as_float(m);
      if (a < kActClampEps) a = kActClampEps;
      s_tok[t] = __fdiv_rn(127.0f, a);
    }
  } else {
#pragma unroll
    for (int t = 0; t < MT; ++t) s_tok[t] = t < c.ntok ? __ldg(c.s_in + c.tok0 + t) : 1.0f;
  }
  if (warp == 0 && lane < MT && lane < c.ntok) {
    float st = s_tok[0];
#pragma unroll
    for (int t = 1; t < MT; ++t)
      if (lane == t) st = s_tok[t];
    tsc_sm[lane] = __fdiv_rn(gamma, st);
    if (FUSED && blockIdx.x == 0) c.s_out[c.tok0 + lane] = st;
  }

  // activations of this lane's words, transposed, plus their sums
  uint32_t xr[J][4][MT];
  int32_t xsum[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) xsum[t] = 0;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int w = wbeg + lane + 32 * j;
    const bool valid = w < wend;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      uint32_t nat[4] = {0u, 0u, 0u, 0u};
      if (valid && t < c.ntok) {
        const int64_t tok = c.tok0 + t;
        if (FUSED) {
          if (onepass) {
            quant16_bf16(raw[kOnePassShape ? j : 0][0], raw[kOnePassShape ? j : 0][1], s_tok[t], nat);
          } else {
            const char* xrow = static_cast<const char*>(c.X) + tok * c.K * (c.x_bf16 ? 2 : 4);
            quant16(xrow, c.x_bf16, 16 * (int64_t)w, s_tok[t], nat);
          }
          if (blockIdx.x == 0 && rg == 0)
            reinterpret_cast<uint4*>(c.xq_out + tok * c.K)[w] = make_uint4(nat[0], nat[1], nat[2], nat[3]);
        } else {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(c.xq_in + tok * c.K) + w);
          nat[0] = v.x;
          nat[1] = v.y;
          nat[2] = v.z;
          nat[3] = v.w;
        }
      }
      uint32_t o[4];
      transpose4x4(nat[0], nat[1], nat[2], nat[3], o);
#pragma unroll
      for (int i = 0; i < 4; ++i) xr[j][i][t] = o[i];
      xsum[t] = __dp4a((int)nat[0], 0x01010101,
                       __dp4a((int)nat[1], 0x01010101,
                              __dp4a((int)nat[2], 0x01010101, __dp4a((int)nat[3], 0x01010101, xsum[t]))));
    }
  }

  const int lane_off = 4 * (wbeg + lane);  // byte offset of this lane's first word in a row
  const bool writer = reduce_writer<V>(lane);
  const int widx = reduce_index<V>(lane);
  const int w_rr = widx / MT, w_t = widx % MT;

  for (int st = 0; st < nstages; ++st) {
    const int slot = st % NS;
    const int rows = min(SR, nrows - st * SR);
    const bool ok = wait_or_abort(&full[slot], (uint32_t)(st / NS) & 1u, c.err, kErrGemvFullWait, abort_flag);
    if (ok) {
      const uint8_t* base = smem + slot * stage_bytes;
      for (int r0 = rg * RI; r0 < rows; r0 += nrg * RI) {
        int32_t a[RI][MT][4];
#pragma unroll
        for (int rr = 0; rr < RI; ++rr)
#pragma unroll
          for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) a[rr][t][i] = 0;
        // one pointer per row (rows past the stage's last valid row read that
        // row again; their sums are discarded), words at immediate offsets.
        // Words past this lane's K slice multiply activations held as zero,
        // and the allocation has slack for reads past the end of a row.
        const uint8_t* rp[RI];
#pragma unroll
        for (int rr = 0; rr < RI; ++rr) rp[rr] = base + min(r0 + rr, rows - 1) * c.row_bytes + lane_off;
#pragma unroll
        for (int j = 0; j < J; ++j) {
          uint32_t P[RI];
#pragma unroll
          for (int rr = 0; rr < RI; ++rr) P[rr] = *reinterpret_cast<const uint32_t*>(rp[rr] + 128 * j);
#pragma unroll
          for (int rr = 0; rr < RI; ++rr)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t m = P[rr] & (0x03030303u << (2 * i));
#pragma unroll
              for (int t = 0; t < MT; ++t) a[rr][t][i] = dp4a_us(m, xr[j][i][t], a[rr][t][i]);
            }
        }
        int32_t v[V];
#pragma unroll
        for (int rr = 0; rr < RI; ++rr)
#pragma unroll
          for (int t = 0; t < MT; ++t)
            v[rr * MT + t] = a[rr][t][0] + (a[rr][t][1] >> 2) + (a[rr][t][2] >> 4) + (a[rr][t][3] >> 6) - xsum[t];
        const int32_t tot = butterfly_sum<V>(v, lane);
        if (writer && r0 + w_rr < rows) atomicAdd(&acc_sm[(st * SR + r0 + w_rr) * MT + w_t], tot);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  consumer_bar();
  if (*abort_flag == 0u) {
    for (int idx = threadIdx.x; idx < nrows * c.ntok; idx += 32 * kConsumerWarps) {
      const int t = idx / nrows, r = idx - t * nrows;
      const int32_t v = acc_sm[r * MT + t];
      const int64_t o = (int64_t)(c.tok0 + t) * c.N + row0 + r;
      c.y[o] = out_act(__fmul_rn(__int2float_rn(v), tsc_sm[t]), c.relu2);
      if (c.acc) c.acc[o] = v;
    }
  }
}

template <int MT, int J, bool FUSED>
cudaError_t launch_one(const GemvCfg& c, int grid, size_t smem, bool pdl, cudaStream_t stream) {
  // four rows per warp iteration where a stage holds enough rows for every row
  // group and the activation registers leave room (J <= 4)
  const bool four = MT == 1 && J <= 4 && c.rows_per_stage >= 4 * (kConsumerWarps / c.kw);
  auto kern = four ? gemv_kernel<MT, J, (MT == 1 ? 4 : 1), FUSED> : gemv_kernel<MT, J, (MT == 1 ? 2 : 1), FUSED>;
  cudaError_t e = set_smem_attrs(kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, c);
}

// Activation registers per lane are J*4*MT.  The limits keep every variant
// within the register budget of three resident CTAs per SM.
constexpr int jmax_for(int mt) { return mt == 1 ? 8 : mt == 2 ? 4 : 2; }

// The smallest instantiated J >= the J a launch needs.
template <int MT, bool FUSED>
cudaError_t dispatch_j(const GemvCfg& c, int J, int grid, size_t smem, bool pdl, cudaStream_t stream) {
  switch (J) {
    case 1: return launch_one<MT, 1, FUSED>(c, grid, smem, pdl, stream);
    case 2: return launch_one<MT, 2, FUSED>(c, grid, smem, pdl, stream);
    default: break;
  }
  if constexpr (MT <= 2) {
    switch (J) {
      case 3: return launch_one<MT, 3, FUSED>(c, grid, smem, pdl, stream);
      case 4: return launch_one<MT, 4, FUSED>(c, grid, smem, pdl, stream);
      default: break;
    }
  }
  if constexpr (MT == 1) {
    switch (J) {
      case 5: return launch_one<MT, 5, FUSED>(c, grid, smem, pdl, stream);
      case 6: return launch_one<MT, 6, FUSED>(c, grid, smem, pdl, stream);
      case 7: return launch_one<MT, 7, FUSED>(c, grid, smem, pdl, stream);
      case 8: return launch_one<MT, 8, FUSED>(c, grid, smem, pdl, stream);
      default: break;
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t run(const ForwardArgs& a, const void* X, bool x_bf16, int8_t* xq_out, float* s_out, bool fused,
                bool pdl, bool test_stall, int num_sms, cudaStream_t stream) {
  GemvCfg c{};
  c.test_stall = test_stall ? 1 : 0;
  c.relu2 = a.relu2 ? 1 : 0;
  c.Wp = a.Wp;
  c.gamma = a.gamma;
  c.xq_in = a.xq;
  c.s_in = a.s;
  c.X = X;
  c.x_bf16 = x_bf16 ? 1 : 0;
  c.xq_out = xq_out;
  c.s_out = s_out;
  c.y = a.y;
  c.acc = a.acc;
  c.err = a.err;
  c.N = a.N;
  c.K = a.K;
  c.row_bytes = (int)(a.K / 4);
  c.words_per_row = (int)(a.K / 16);

  // CTAs per SM: two, except on the fused path when one CTA per SM still gets
  // its whole share of the weights in a single stage (decode-sized matrices):
  // there every CTA repeats the activation quantisation, and fewer CTAs finish
  // sooner (measured on B300).
  const bool small = (int64_t)a.N * c.row_bytes <= (int64_t)num_sms * kStageBytesTarget;
  const int64_t max_grid = (int64_t)num_sms * ((fused && small) ? 1 : kCtasPerSm);
  int grid = (int)(a.N < max_grid ? a.N : max_grid);
  c.rows_per_cta = (int)((a.N + grid - 1) / grid);
  grid = (int)((a.N + c.rows_per_cta - 1) / c.rows_per_cta);
  int sr = kStageBytesTarget / c.row_bytes;
  if (sr < 1) sr = 1;
  if (sr > c.rows_per_cta) sr = c.rows_per_cta;
  c.rows_per_stage = sr;
  const int max_stages = (c.rows_per_cta + sr - 1) / sr;
  c.nslots = max_stages < kStages ? max_stages : kStages;

  // tokens per pass: 4, 2 or 1 (<= M), limited by the activation registers
  int mt = a.M >= 4 ? 4 : a.M >= 2 ? 2 : 1;
  while (mt > 1 && (c.words_per_row + 32 * kConsumerWarps - 1) / (32 * kConsumerWarps) > jmax_for(mt)) mt /= 2;
  int kw = 1;
  while (kw < kConsumerWarps && (c.words_per_row + 32 * kw - 1) / (32 * kw) > jmax_for(mt)) kw *= 2;
  // one token: at most 4 words per lane where possible (the one-pass fused
  // prologue needs it, and four rows per iteration fit the registers)
  if (mt == 1)
    while (kw < kConsumerWarps && (c.words_per_row + 32 * kw - 1) / (32 * kw) > 4) kw *= 2;
  c.kw = kw;
  c.words_per_warp = (c.words_per_row + c.kw - 1) / c.kw;
  const int J = (c.words_per_warp + 31) / 32;
  if (J > jmax_for(mt)) return cudaErrorInvalidValue;  // K beyond the GEMV's register budget
  // slack: a lane may read up to 32 * J * kw words past the end of the last row
  const size_t slack = (size_t)128 * J * c.kw;
  const size_t smem = (size_t)c.nslots * c.rows_per_stage * c.row_bytes + 2 * kStages * sizeof(uint64_t) +
                      (size_t)c.rows_per_cta * mt * sizeof(int32_t) + (kConsumerWarps + 1) * mt * 4 + 16 + slack;

  for (int64_t t0 = 0; t0 < a.M; t0 += mt) {
    c.tok0 = (int)t0;
    c.ntok = (int)(a.M - t0 < mt ? a.M - t0 : mt);
    cudaError_t e;
    if (fused) {
      if (mt == 4) e = dispatch_j<4, true>(c, J, grid, smem, pdl, stream);
      else if (mt == 2) e = dispatch_j<2, true>(c, J, grid, smem, pdl, stream);
      else e = dispatch_j<1, true>(c, J, grid, smem, pdl, stream);
    } else {
      if (mt == 4) e = dispatch_j<4, false>(c, J, grid, smem, pdl, stream);
      else if (mt == 2) e = dispatch_j<2, false>(c, J, grid, smem, pdl, stream);
      else e = dispatch_j<1, false>(c, J, grid, smem, pdl, stream);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv(const ForwardArgs& a, int num_sms, cudaStream_t stream, bool pdl) {
  return run(a, nullptr, false, nullptr, nullptr, false, pdl, false, num_sms, stream);
}

cudaError_t launch_gemv_fused(const ForwardArgs& a, const void* X, bool x_bf16, int8_t* xq_out, float* s_out,
                              bool pdl, bool test_stall, int num_sms, cudaStream_t stream) {
  return run(a, X, x_bf16, xq_out, s_out, true, pdl, test_stall, num_sms, stream);
}

}  // namespace bl
