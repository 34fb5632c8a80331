// quant.cu -- per-token absmax int8 quantisation of activations ("activations
// at 8 bits": anthology note-168 on arXiv 2402.17764, "What it does").
//
//   a    = max(max_k |x[m,k]|, 1e-5)         (clamp: an all-zero token stays finite)
//   s[m] = fp32(127 / a)                     (one IEEE division)
//   x_q  = clip(rint(fp32(x * s[m])), -128, 127)   (rint = round half to even)
//
// One CTA per token row.  Pass 1 reduces max|x| over the row with 128-bit
// loads (as fp32 bit patterns: for non-negative floats the unsigned order is
// the numeric order, so the reduction is exact and order-free); pass 2 reads
// the row again (from L1/L2) and writes x_q.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "sumsq_exact.cuh"

namespace bl {
namespace {

constexpr float kActClampEps = 1e-5f;

__device__ __forceinline__ uint32_t abs_bits_bf16x2(uint32_t w) {
  return max((w << 16) & 0x7fff0000u, w & 0x7fff0000u);
}

__device__ __forceinline__ uint32_t q8(float x, float s) {
  int q = __float2int_rn(__fmul_rn(x, s));
  q = min(max(q, -128), 127);
  return (uint32_t)q & 0xffu;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Where the fp8 GEMM's operand goes (OUT == 2): the tiled layout of
// x8_group_offset, tokens in tiles of BN, nkb 512-k blocks, M real tokens.
// cnt / ncnt also serve OUT == 1 (the stream-K GEMM's counters).
struct X8Out {
  uint8_t* x8;
  uint32_t* cnt;  // arrival counters, zeroed by block 0 (OUT != 0)
  int ncnt;
  int64_t M, nkb;
  int BN;
  int32_t* sx;  // OUT == 2: every token's x8_sum_parts(K) partial sums of int8 activations (0 for padding tokens)
};

// Clusters of CTAs sharing one token row (a launch without clusters is a
// cluster of one): rank, size, barrier, and a 32-bit load from a peer's
// shared memory at the same offset as `local`.
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cl_load_peer(const void* local, uint32_t rank) {
  uint32_t ra, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

// OUT: 0 x_q and s only; 1 also the fp16 operand of the f16 GEMM (x16,
// M x K halves); 2 also the e4m3 operand of the fp8 GEMM: the grid then has a
// CTA for every token of the last tile, and the CTAs of tokens past M (and
// every CTA for k past K in the last block) write zeros.
// A row may be shared by a cluster of up to 8 CTAs (launched with cluster
// dimensions): each takes a contiguous slice of the row, and the slices'
// maxima (and, for OUT == 2, activation sums) are exchanged through
// distributed shared memory; max and integer sums do not depend on the split.
template <bool BF16, int OUT>
__global__ void __launch_bounds__(1024) quant_act_kernel(const void* __restrict__ X, int64_t K, bool vec,
                                                         int8_t* __restrict__ xq, float* __restrict__ s,
                                                         uint4* __restrict__ xop, const X8Out o8) {
  constexpr int kEsize = BF16 ? 2 : 4;
  const uint32_t S = cl_size(), rk = S > 1 ? cl_rank() : 0u;  // CTAs per row, this CTA's slice
  const int64_t m = S > 1 ? blockIdx.x / S : blockIdx.x;
  pdl_launch_dependents();  // a dependent GEMV may start streaming its weights now
  if (OUT != 0 && blockIdx.x == 0)
    for (int i = threadIdx.x; i < o8.ncnt; i += blockDim.x) o8.cnt[i] = 0u;
  // slice [lo, hi) of n items (n * 8 < 2^32: K <= 2^24); no division for an unsplit row
  auto slice_lo = [&](int64_t n) -> int64_t { return S > 1 ? (uint32_t)n * rk / S : 0; };
  auto slice_hi = [&](int64_t n) -> int64_t { return S > 1 ? (uint32_t)n * (rk + 1u) / S : n; };
  if (OUT == 2) {
    const int64_t kpad = o8.nkb * kX8Block;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t k16 = (m < o8.M ? K : 0) + 16 * ((int64_t)threadIdx.x + (int64_t)rk * blockDim.x); k16 < kpad;
         k16 += 16 * (int64_t)blockDim.x * S) {
      *reinterpret_cast<uint4*>(o8.x8 + x8_group_offset(m, k16, 0, o8.BN, o8.nkb)) = z;
      *reinterpret_cast<uint4*>(o8.x8 + x8_group_offset(m, k16, 1, o8.BN, o8.nkb)) = z;
    }
    if (m >= o8.M) {  // a padding token of the last tile: zeros only (the whole cluster, before any barrier)
      if (rk == 0)
        for (int pc = threadIdx.x; pc < x8_sum_parts(K); pc += blockDim.x) o8.sx[m * x8_sum_parts(K) + pc] = 0;
      return;
    }
  }
  const char* row = static_cast<const char*>(X) + m * K * kEsize;
  int8_t* out = xq + m * K;
  const int tid = threadIdx.x, nt = blockDim.x;

  uint32_t amax = 0;
  if (vec) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int64_t nch = K * kEsize / 16;
    for (int64_t c = slice_lo(nch) + tid, c_end = slice_hi(nch); c < c_end; c += nt) {
      const uint4 v = __ldg(r4 + c);
      if (BF16) {
        amax = max(amax, max(max(abs_bits_bf16x2(v.x), abs_bits_bf16x2(v.y)),
                             max(abs_bits_bf16x2(v.z), abs_bits_bf16x2(v.w))));
      } else {
        amax = max(amax, max(max(v.x & 0x7fffffffu, v.y & 0x7fffffffu), max(v.z & 0x7fffffffu, v.w & 0x7fffffffu)));
      }
    }
  } else {
    for (int64_t k = slice_lo(K) + tid, k_end = slice_hi(K); k < k_end; k += nt) {
      uint32_t b = BF16 ? ((uint32_t)reinterpret_cast<const uint16_t*>(row)[k] << 16)
                        : reinterpret_cast<const uint32_t*>(row)[k];
      amax = max(amax, b & 0x7fffffffu);
    }
  }
  __shared__ uint32_t red[32];
  __shared__ uint32_t cl_max;  // this CTA's slice maximum, read by the other CTAs of the row
  amax = __reduce_max_sync(0xffffffffu, amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid < 32) {
    uint32_t v = tid < (nt >> 5) ? red[tid] : 0u;
    v = __reduce_max_sync(0xffffffffu, v);
    if (tid == 0) red[0] = cl_max = v;
  }
  if (S > 1) {
    cl_barrier();  // every slice maximum is written
    if (tid == 0) {
      uint32_t v = 0u;
      for (uint32_t q = 0; q < S; ++q) v = max(v, cl_load_peer(&cl_max, q));
      red[0] = v;
    }
  }
  __syncthreads();
  float a = __uint_as_float(red[0]);
  if (a < kActClampEps) a = kActClampEps;
  const float sm = __fdiv_rn(127.0f, a);
  if (tid == 0 && rk == 0) s[m] = sm;

  if (OUT != 0) {
    // groups of 16 activations: x_q (natural order) and the GEMM's operand:
    // fp16 in the order p = 4i + j within the group, or the two e4m3 rows;
    // K % 16 == 0
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    int xsum = 0;
    for (int64_t g = slice_lo(K / 16) + tid, g_end = slice_hi(K / 16); g < g_end; g += nt) {
      uint32_t nat[4];
      if (BF16) {
        const uint4 a = __ldg(r4 + 2 * g), b = __ldg(r4 + 2 * g + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          nat[i] = q8(bf16_lo(w[2 * i]), sm) | (q8(bf16_hi(w[2 * i]), sm) << 8) | (q8(bf16_lo(w[2 * i + 1]), sm) << 16) |
                   (q8(bf16_hi(w[2 * i + 1]), sm) << 24);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = __ldg(r4 + 4 * g + i);
          nat[i] = q8(__uint_as_float(v.x), sm) | (q8(__uint_as_float(v.y), sm) << 8) |
                   (q8(__uint_as_float(v.z), sm) << 16) | (q8(__uint_as_float(v.w), sm) << 24);
        }
      }
      const uint4 q4 = make_uint4(nat[0], nat[1], nat[2], nat[3]);
      reinterpret_cast<uint4*>(out)[g] = q4;
      if (OUT == 1) {
        uint32_t h[8];
        convert_x16_f16(q4, h);
        uint4* xo = xop + m * (K / 8);
        xo[2 * g] = make_uint4(h[0], h[1], h[2], h[3]);
        xo[2 * g + 1] = make_uint4(h[4], h[5], h[6], h[7]);
      } else {
        uint4 hi, lo;
        x8_rows16(q4, &hi, &lo);
        *reinterpret_cast<uint4*>(o8.x8 + x8_group_offset(m, 16 * g, 0, o8.BN, o8.nkb)) = hi;
        *reinterpret_cast<uint4*>(o8.x8 + x8_group_offset(m, 16 * g, 1, o8.BN, o8.nkb)) = lo;
        xsum += sum16_i8(q4);
      }
    }
    if (OUT == 2) {  // the whole row's sum in the first of the token's partial sums, zeros in the rest
      __shared__ int32_t cl_sum;  // this CTA's slice sum, read by rank 0
      if (rk == 0)
        for (int pc = 1 + tid; pc < x8_sum_parts(K); pc += nt) o8.sx[m * x8_sum_parts(K) + pc] = 0;
      block_sum_store(xsum, S > 1 ? &cl_sum : o8.sx + m * x8_sum_parts(K));
      if (S > 1) {
        cl_barrier();  // every slice sum is written
        if (rk == 0 && tid == 0) {
          int32_t v = 0;
          for (uint32_t q = 0; q < S; ++q) v += (int32_t)cl_load_peer(&cl_sum, q);
          o8.sx[m * x8_sum_parts(K)] = v;
        }
      }
    }
  } else if (vec) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int64_t nch = K * kEsize / 16;
    for (int64_t c = slice_lo(nch) + tid, c_end = slice_hi(nch); c < c_end; c += nt) {
      const uint4 v = __ldg(r4 + c);
      if (BF16) {
        uint2 o;
        o.x = q8(bf16_lo(v.x), sm) | (q8(bf16_hi(v.x), sm) << 8) | (q8(bf16_lo(v.y), sm) << 16) |
              (q8(bf16_hi(v.y), sm) << 24);
        o.y = q8(bf16_lo(v.z), sm) | (q8(bf16_hi(v.z), sm) << 8) | (q8(bf16_lo(v.w), sm) << 16) |
              (q8(bf16_hi(v.w), sm) << 24);
        reinterpret_cast<uint2*>(out)[c] = o;
      } else {
        const uint32_t o = q8(__uint_as_float(v.x), sm) | (q8(__uint_as_float(v.y), sm) << 8) |
                           (q8(__uint_as_float(v.z), sm) << 16) | (q8(__uint_as_float(v.w), sm) << 24);
        reinterpret_cast<uint32_t*>(out)[c] = o;
      }
    }
  } else {
    for (int64_t k = slice_lo(K) + tid, k_end = slice_hi(K); k < k_end; k += nt) {
      const float x = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(row)[k] << 16)
                           : reinterpret_cast<const float*>(row)[k];
      out[k] = (int8_t)q8(x, sm);
    }
  }
  if (S > 1) cl_barrier();  // no CTA leaves while another may still read its shared memory
}

// Sub-layer RMS normalisation, then the quantisation of the normalised row
// (the normalisation BitNet b1.58 2B4T adds inside each sub-layer: yousumm.com
// transcript, the paragraph after the poker-chip analogy).  Per token:
//   ms  = mean(x^2), exact, rounded once to fp32 (sumsq_exact.cuh)
//   r   = fp32 sqrt(fp32(ms + eps))
//   x_n = fp32(fp32(x * g) / r)
//   s   = 127 / max(max|x_n|, 1e-5),  x_q = clip(rint(fp32(x_n * s)), -128, 127)
// Division by r > 0 rounds monotonically, so max|x_n| = fp32(max|x * g| / r).
// One CTA per token (at least one full warp: the finish is warp-wide), three
// passes over the row, each a rolled loop over 16-byte chunks (the row is
// read from DRAM once, then from L1):
//   1. max|x * g| and max|x| (order-free, on fp32 bit patterns); max|x| fixes
//      the top exponent group of the squares;
//   2. the exact sum of x^2;
//   3. after one warp has finished ms, r and s: the codes of x_n.
// The code stays small on purpose: each CTA runs it once, on whichever SM it
// lands, so instruction fetch, not arithmetic, sets a short row's time.
// Rows or gains that are not 16-byte aligned take an element-wise path with
// the same arithmetic.

__device__ __forceinline__ void block_reduce_max2(uint32_t& a, uint32_t& b, uint32_t* red) {
  const int tid = threadIdx.x, nw = blockDim.x >> 5;
  a = __reduce_max_sync(0xffffffffu, a);
  b = __reduce_max_sync(0xffffffffu, b);
  if ((tid & 31) == 0) {
    red[tid >> 5] = a;
    red[32 + (tid >> 5)] = b;
  }
  __syncthreads();
  if (tid < 32) {
    uint32_t u = tid < nw ? red[tid] : 0u, v = tid < nw ? red[32 + tid] : 0u;
    u = __reduce_max_sync(0xffffffffu, u);
    v = __reduce_max_sync(0xffffffffu, v);
    if (tid == 0) {
      red[64] = u;
      red[65] = v;
    }
  }
  __syncthreads();
  a = red[64];
  b = red[65];
}

template <bool BF16>
__device__ __forceinline__ void unpack_chunk(const uint4 v, float* x) {
  if (BF16) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_lo(w[i]);
      x[2 * i + 1] = bf16_hi(w[i]);
    }
  } else {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
}

// OUT as in quant_act_kernel: 0 x_q and s only; 1 also the fp16 GEMM operand;
// 2 also the fp8 GEMM operand (the grid then covers every token of the last
// tile; padding tokens write zeros only).  OUT != 0 needs vec and K % 16 == 0.
template <bool BF16, int OUT>
__global__ void __launch_bounds__(1024) rmsnorm_quant_act_kernel(const void* __restrict__ X, int64_t K, bool vec,
                                                                 const float* __restrict__ gain, float eps,
                                                                 unsigned long long recip_k, int8_t* __restrict__ xq,
                                                                 float* __restrict__ s, uint4* __restrict__ xop,
                                                                 const X8Out o8) {
  constexpr int kEsize = BF16 ? 2 : 4;
  constexpr int kPer = 16 / kEsize;  // elements per 16-byte chunk
  const int64_t m = blockIdx.x;
  if (OUT != 0 && blockIdx.x == 0)
    for (int i = threadIdx.x; i < o8.ncnt; i += blockDim.x) o8.cnt[i] = 0u;
  if (OUT == 2) {
    const int64_t kpad = o8.nkb * kX8Block;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t k16 = (m < o8.M ? K : 0) + 16 * (int64_t)threadIdx.x; k16 < kpad; k16 += 16 * (int64_t)blockDim.x) {
      *reinterpret_cast<uint4*>(o8.x8 + x8_group_offset(m, k16, 0, o8.BN, o8.nkb)) = z;
      *reinterpret_cast<uint4*>(o8.x8 + x8_group_offset(m, k16, 1, o8.BN, o8.nkb)) = z;
    }
    if (m >= o8.M) {  // a padding token of the last tile: zeros only (whole CTA, before any barrier)
      for (int pc = threadIdx.x; pc < x8_sum_parts(K); pc += blockDim.x) o8.sx[m * x8_sum_parts(K) + pc] = 0;
      return;
    }
  }
  const char* row = static_cast<const char*>(X) + m * K * kEsize;
  const uint4* row4 = reinterpret_cast<const uint4*>(row);
  const float4* gain4 = reinterpret_cast<const float4*>(gain);
  int8_t* out = xq + m * K;
  const int tid = threadIdx.x, nt = blockDim.x;
  __shared__ uint32_t red[66];
  __shared__ SqBuckets sb;
  __shared__ float fin[2];  // r, s
  sq_clear(&sb);

  auto load_gain = [&](int64_t c, float (&g)[kPer]) {
    if (gain) {
#pragma unroll
      for (int h = 0; h < kPer / 4; ++h) {
        const float4 q = __ldg(gain4 + c * (kPer / 4) + h);
        g[4 * h] = q.x;
        g[4 * h + 1] = q.y;
        g[4 * h + 2] = q.z;
        g[4 * h + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kPer; ++i) g[i] = 1.0f;
    }
  };
  auto load = [&](int64_t k) -> float {
    return BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(row)[k] << 16)
                : reinterpret_cast<const float*>(row)[k];
  };
  const int64_t nch = vec ? K / kPer : 0;

  // pass 1: max|x * g| and max|x|
  uint32_t amax_t = 0, amax_x = 0;
  if (vec) {
#pragma unroll 1
    for (int64_t c = tid; c < nch; c += nt) {
      float x[kPer], g[kPer];
      unpack_chunk<BF16>(__ldg(row4 + c), x);
      load_gain(c, g);
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        amax_x = max(amax_x, __float_as_uint(x[i]) & 0x7fffffffu);
        amax_t = max(amax_t, __float_as_uint(__fmul_rn(x[i], g[i])) & 0x7fffffffu);
      }
    }
  } else {
#pragma unroll 1
    for (int64_t k = tid; k < K; k += nt) {
      const float x = load(k);
      const float t = gain ? __fmul_rn(x, __ldg(gain + k)) : x;
      amax_x = max(amax_x, __float_as_uint(x) & 0x7fffffffu);
      amax_t = max(amax_t, __float_as_uint(t) & 0x7fffffffu);
    }
  }
  block_reduce_max2(amax_t, amax_x, red);  // its barriers also order sq_clear before the adds

  // pass 2: the exact sum of x^2
  SqAcc sq(sq_group(amax_x));
  if (vec) {
#pragma unroll 1
    for (int64_t c = tid; c < nch; c += nt) {
      float x[kPer];
      unpack_chunk<BF16>(__ldg(row4 + c), x);
#pragma unroll
      for (int i = 0; i < kPer; ++i) sq.add(x[i], &sb);
    }
  } else {
#pragma unroll 1
    for (int64_t k = tid; k < K; k += nt) sq.add(load(k), &sb);
  }
  sq.flush_warp(&sb);
  __syncthreads();
  if (tid < 32) {
    const float ms = sq_mean_f32(&sb, (uint32_t)K, recip_k);  // the whole warp
    const float r = __fsqrt_rn(__fadd_rn(ms, eps));
    float a = __fdiv_rn(__uint_as_float(amax_t), r);
    if (a < kActClampEps) a = kActClampEps;
    const float sg = __fdiv_rn(127.0f, a);
    if (tid == 0) {
      fin[0] = r;
      fin[1] = sg;
      s[m] = sg;
    }
  }
  __syncthreads();
  const float r = fin[0], sg = fin[1];

  // pass 3: codes of x_n = fp32(x * g) / r
  if (OUT != 0) {
    // one 16-element group per thread: x_q (natural order) and the GEMM's operand
    int xsum = 0;
#pragma unroll 1
    for (int64_t gq = tid; gq < K / 16; gq += nt) {
      uint32_t nat[4];
#pragma unroll
      for (int c2 = 0; c2 < 16 / kPer; ++c2) {
        const int64_t c = gq * (16 / kPer) + c2;
        float x[kPer], g[kPer];
        unpack_chunk<BF16>(__ldg(row4 + c), x);
        load_gain(c, g);
        uint32_t q[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) q[i] = q8(__fdiv_rn(__fmul_rn(x[i], g[i]), r), sg);
#pragma unroll
        for (int w = 0; w < kPer / 4; ++w)
          nat[c2 * (kPer / 4) + w] = q[4 * w] | (q[4 * w + 1] << 8) | (q[4 * w + 2] << 16) | (q[4 * w + 3] << 24);
      }
      const uint4 q4 = make_uint4(nat[0], nat[1], nat[2], nat[3]);
      reinterpret_cast<uint4*>(out)[gq] = q4;
      if (OUT == 1) {
        uint32_t h[8];
        convert_x16_f16(q4, h);
        uint4* xo = xop + m * (K / 8);
        xo[2 * gq] = make_uint4(h[0], h[1], h[2], h[3]);
        xo[2 * gq + 1] = make_uint4(h[4], h[5], h[6], h[7]);
      } else {
        uint4 hi, lo;
        x8_rows16(q4, &hi, &lo);
        *reinterpret_cast<uint4*>(o8.x8 + x8_group_offset(m, 16 * gq, 0, o8.BN, o8.nkb)) = hi;
        *reinterpret_cast<uint4*>(o8.x8 + x8_group_offset(m, 16 * gq, 1, o8.BN, o8.nkb)) = lo;
        xsum += sum16_i8(q4);
      }
    }
    if (OUT == 2) {  // the whole row's sum in the first of the token's partial sums, zeros in the rest
      for (int pc = 1 + tid; pc < x8_sum_parts(K); pc += nt) o8.sx[m * x8_sum_parts(K) + pc] = 0;
      block_sum_store(xsum, o8.sx + m * x8_sum_parts(K));
    }
  } else if (vec) {
#pragma unroll 1
    for (int64_t c = tid; c < nch; c += nt) {
      float x[kPer], g[kPer];
      unpack_chunk<BF16>(__ldg(row4 + c), x);
      load_gain(c, g);  // the gain row is shared by every token: an L1 hit
      uint32_t q[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) q[i] = q8(__fdiv_rn(__fmul_rn(x[i], g[i]), r), sg);
      if (BF16) {
        uint2 o;
        o.x = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
        o.y = q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24);
        reinterpret_cast<uint2*>(out)[c] = o;
      } else {
        reinterpret_cast<uint32_t*>(out)[c] = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
      }
    }
  } else {
#pragma unroll 1
    for (int64_t k = tid; k < K; k += nt) {
      const float x = load(k);
      const float t = gain ? __fmul_rn(x, __ldg(gain + k)) : x;
      out[k] = (int8_t)q8(__fdiv_rn(t, r), sg);
    }
  }
}

// fp32(x * s) rounded half to even by one fp32 add of 1.5 * 2^23: while
// |x * s| < 2^22 the sum is 1.5 * 2^23 + rint(x * s) exactly (its ulp is 1,
// and 1.5 * 2^23 is even, so ties go to the even integer), and the low byte
// of its bits is the integer's two's-complement low byte.  For finite inputs
// |x * s| <= 127 * (1 + 2^-24)^2, so this is the code of q8 (whose clamp never
// acts) without the quarter-rate float-to-int conversion.
__device__ __forceinline__ uint32_t q8_bits(float x, float s) {
  return __float_as_uint(__fadd_rn(__fmul_rn(x, s), 12582912.0f));
}

// low bytes of a, b, c, d -> bytes 0..3 of one word
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

// Many tokens: the same normalisation and quantisation with one warp per row
// (kRmsRowWarps rows per CTA).  With one CTA per row, every row waits on three
// block barriers and on the one-warp finish while its other warps idle, and an
// SM holds only a few rows; a warp per row needs no block barrier (the finish
// is warp-wide already) and keeps many rows in flight per SM.  Each warp has
// its own buckets; the passes, their arithmetic and therefore x_q, s and the
// operand are those of rmsnorm_quant_act_kernel bit for bit (its codes via
// q8_bits: |x_n| <= max|x_n| = a and s = 127 / a bound |x_n * s| as there).
// Needs the 16-byte path (rows, gain and x_q aligned; OUT == 1: K % 16 == 0).
constexpr int kRmsRowWarps = 4;
// It serves from 1536 tokens with rows of at most 8 KB, where it measured
// faster (warp per row / CTA per row: 1536 x 2560 bf16 21.4 / 26.8 us,
// 2048 x 2560 24.8 / 33.7 us, 8192 x 2560 81.5 / 122 us, 2048 x 4096
// 37.2 / 46.8 us, 2048 x 2048 fp32 24.3 / 33.9 us).  With fewer rows per SM,
// or longer rows, one CTA per row is faster (1024 x 2560 bf16 19.5 / 18.5 us,
// 512 x 2560 18.7 / 10.8 us, 600 x 28672 206 / 86 us; 2048 x 6912 fp32
// equal): the three passes take an estimated 60 instructions per element
// (the IEEE division and the exact square sum), so a lone warp per row is
// issue-bound.
constexpr int64_t kRmsRowWarpsMinM = 1536;
constexpr int64_t kRmsRowWarpsMaxRowBytes = 8192;
__host__ __device__ constexpr bool rms_row_warps_serve(int64_t M, int64_t row_bytes) {
  return M >= kRmsRowWarpsMinM && row_bytes <= kRmsRowWarpsMaxRowBytes;
}

template <bool BF16, int OUT>
__global__ void __launch_bounds__(32 * kRmsRowWarps) rmsnorm_quant_rows_kernel(
    const void* __restrict__ X, int64_t M, int64_t K, const float* __restrict__ gain, float eps,
    unsigned long long recip_k, int8_t* __restrict__ xq, float* __restrict__ s, uint4* __restrict__ xop,
    uint32_t* __restrict__ cnt, int ncnt) {
  constexpr int kEsize = BF16 ? 2 : 4;
  constexpr int kPer = 16 / kEsize;  // elements per 16-byte chunk
  static_assert(kSqGroups == 32, "one bucket per lane");
  if (OUT != 0 && blockIdx.x == 0)
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0u;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t m = (int64_t)blockIdx.x * kRmsRowWarps + w;
  if (m >= M) return;  // the whole warp (no block barrier follows)
  __shared__ SqBuckets sbs[kRmsRowWarps];
  SqBuckets* sb = &sbs[w];
  sb->lo[lane] = 0;
  sb->hi[lane] = 0;
  __syncwarp();

  const uint4* row4 = reinterpret_cast<const uint4*>(static_cast<const char*>(X) + m * K * kEsize);
  const float4* gain4 = reinterpret_cast<const float4*>(gain);
  int8_t* out = xq + m * K;
  auto load_gain = [&](int64_t c, float (&g)[kPer]) {
    if (gain) {
#pragma unroll
      for (int h = 0; h < kPer / 4; ++h) {
        const float4 q = __ldg(gain4 + c * (kPer / 4) + h);
        g[4 * h] = q.x;
        g[4 * h + 1] = q.y;
        g[4 * h + 2] = q.z;
        g[4 * h + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kPer; ++i) g[i] = 1.0f;
    }
  };
  const int64_t nch = K / kPer;

  // pass 1: max|x * g| and max|x| (unrolled: several chunks' loads in flight)
  uint32_t amax_t = 0, amax_x = 0;
#pragma unroll 4
  for (int64_t c = lane; c < nch; c += 32) {
    float x[kPer], g[kPer];
    unpack_chunk<BF16>(__ldg(row4 + c), x);
    load_gain(c, g);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      amax_x = max(amax_x, __float_as_uint(x[i]) & 0x7fffffffu);
      amax_t = max(amax_t, __float_as_uint(__fmul_rn(x[i], g[i])) & 0x7fffffffu);
    }
  }
  amax_t = __reduce_max_sync(0xffffffffu, amax_t);
  amax_x = __reduce_max_sync(0xffffffffu, amax_x);

  // pass 2: the exact sum of x^2
  SqAcc sq(sq_group(amax_x));
#pragma unroll 4
  for (int64_t c = lane; c < nch; c += 32) {
    float x[kPer];
    unpack_chunk<BF16>(__ldg(row4 + c), x);
#pragma unroll
    for (int i = 0; i < kPer; ++i) sq.add(x[i], sb);
  }
  sq.flush_warp(sb);
  __syncwarp();  // every lane's bucket adds are visible to the finish
  const float ms = sq_mean_f32(sb, (uint32_t)K, recip_k);
  const float r = __fsqrt_rn(__fadd_rn(ms, eps));
  float a = __fdiv_rn(__uint_as_float(amax_t), r);
  if (a < kActClampEps) a = kActClampEps;
  const float sg = __fdiv_rn(127.0f, a);
  if (lane == 0) s[m] = sg;

  // pass 3: codes of x_n = fp32(x * g) / r
  if (OUT == 1) {
    // one 16-element group per lane: x_q (natural order) and the fp16 operand
    uint4* xo = xop + m * (K / 8);
#pragma unroll 2
    for (int64_t gq = lane; gq < K / 16; gq += 32) {
      uint32_t nat[4];
#pragma unroll
      for (int c2 = 0; c2 < 16 / kPer; ++c2) {
        const int64_t c = gq * (16 / kPer) + c2;
        float x[kPer], g[kPer];
        unpack_chunk<BF16>(__ldg(row4 + c), x);
        load_gain(c, g);
        uint32_t q[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) q[i] = q8_bits(__fdiv_rn(__fmul_rn(x[i], g[i]), r), sg);
#pragma unroll
        for (int v = 0; v < kPer / 4; ++v)
          nat[c2 * (kPer / 4) + v] = pack_low_bytes(q[4 * v], q[4 * v + 1], q[4 * v + 2], q[4 * v + 3]);
      }
      const uint4 q4 = make_uint4(nat[0], nat[1], nat[2], nat[3]);
      reinterpret_cast<uint4*>(out)[gq] = q4;
      uint32_t h[8];
      convert_x16_f16(q4, h);
      xo[2 * gq] = make_uint4(h[0], h[1], h[2], h[3]);
      xo[2 * gq + 1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  } else {
#pragma unroll 4
    for (int64_t c = lane; c < nch; c += 32) {
      float x[kPer], g[kPer];
      unpack_chunk<BF16>(__ldg(row4 + c), x);
      load_gain(c, g);
      uint32_t q[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) q[i] = q8_bits(__fdiv_rn(__fmul_rn(x[i], g[i]), r), sg);
      if (BF16)
        reinterpret_cast<uint2*>(out)[c] = make_uint2(pack_low_bytes(q[0], q[1], q[2], q[3]),
                                                      pack_low_bytes(q[4], q[5], q[6], q[7]));
      else
        reinterpret_cast<uint32_t*>(out)[c] = pack_low_bytes(q[0], q[1], q[2], q[3]);
    }
  }
}

// ---- many tokens: rows staged in shared memory, one team of warps per row -
//
// With one CTA per row, every CTA on an SM loads, reduces and quantises in
// step, so DRAM idles while rows are being quantised and the last wave runs
// mostly empty.  Here each team of T warps (T = 1, 2, 4 or 8) of a persistent
// grid owns rows gt, gt + GT, ... (GT teams in the grid).  The team's leader
// keeps the next `stages` rows in flight as 1-D bulk copies into the team's
// shared-memory ring; thread t of the team takes the 16-byte chunks t,
// t + 32T, ... of the staged row (consecutive lanes read consecutive chunks:
// no bank conflicts).  The row maximum is a warp reduction, then (T > 1) a
// named barrier over the team.  x_q and s are those of quant_act_kernel bit
// for bit (finite inputs).

struct RowQuantArgs {
  const char* X;  // [M, K] rows, row_bytes = K * element size, 16-byte aligned
  int64_t M, K;
  int8_t* xq;  // [M, K], 16-byte aligned
  float* s;
  uint32_t* err;  // device error word
  uint32_t row_bytes;
  int stages;  // ring depth per team
  int team;    // warps per row
  int stall;   // test hook: no row copies are issued, so the bounded waits expire
};

constexpr int kRowWarpsMax = 16;
constexpr uint32_t kRowBarBytes = 1024;  // mbarriers and per-team flags at the start of shared memory

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <bool BF16>
__global__ void __launch_bounds__(kRowWarpsMax * 32) quant_rows_staged_kernel(const RowQuantArgs a) {
  constexpr int kPer = BF16 ? 8 : 4;  // elements per 16-byte chunk
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint32_t red_max[kRowWarpsMax];  // per warp: max|x| bits of the current row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int T = a.team, nteams = nwarps / T;
  const int team = warp / T, tt = (warp % T) * 32 + lane, TT = T * 32;
  const bool leader = tt == 0;
  const int S = a.stages;
  const int64_t K = a.K, nch = K / kPer;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + team * S;
  volatile int* flag = reinterpret_cast<volatile int*>(smem + kRowBarBytes - 4 * kRowWarpsMax) + team;
  unsigned char* ring = smem + kRowBarBytes + (size_t)team * S * a.row_bytes;
  auto team_sync = [&]() {
    if (T > 1) asm volatile("bar.sync %0, %1;" ::"r"(team + 1), "r"(TT) : "memory");
    else __syncwarp();
  };

  if (leader) {
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    fence_mbarrier_init();
  }
  __syncthreads();

  const int64_t gt = (int64_t)blockIdx.x * nteams + team, GT = (int64_t)gridDim.x * nteams;
  const int64_t nrows = gt < a.M ? (a.M - 1 - gt) / GT + 1 : 0;
  int64_t issued = 0;  // rows 0 .. issued - 1 have been copied for (leader only)
  auto issue = [&](int64_t i, int st) {
    const int64_t m = gt + i * GT;
    mbar_arrive_expect_tx(&bars[st], a.row_bytes);
    bulk_g2s(ring + (size_t)st * a.row_bytes, a.X + m * (int64_t)a.row_bytes, a.row_bytes, &bars[st]);
    issued = i + 1;
  };
  if (leader && !a.stall)
    for (int i = 0; i < S && i < nrows; ++i) issue(i, i);

  int st = 0, prev_st = 0;
  uint32_t phase = 0;
  for (int64_t i = 0; i < nrows; ++i) {
    // the leader waits for the row (bounded) and posts the outcome; after the
    // team barrier every thread of the team has also finished row i - 1
    if (leader) *flag = mbar_wait_bounded(&bars[st], phase, a.err, kErrQuantWait) ? 1 : 0;
    team_sync();
    const bool ok = *flag != 0;
    if (leader && i >= 1 && i - 1 + S < nrows) {
      fence_proxy_async_smem();  // order the team's generic-proxy reads before the async overwrite
      issue(i - 1 + S, prev_st);
    }
    if (!ok) {
      // give up: let every copy still in flight into this team's ring (rows
      // i .. issued - 1, the refill above included) land, each wait bounded,
      // before the CTA's shared memory is released
      if (leader) {
        int sj = st;
        uint32_t pj = phase;
        for (int64_t j = i; j < issued; ++j) {
          mbar_wait_bounded(&bars[sj], pj, a.err, kErrQuantWait);
          if (++sj == S) {
            sj = 0;
            pj ^= 1u;
          }
        }
      }
      return;
    }
    mbar_try_wait(smem_u32(&bars[st]), phase);  // complete: this thread's acquire of the copied row
    const int64_t m = gt + i * GT;
    const uint4* buf = reinterpret_cast<const uint4*>(ring + (size_t)st * a.row_bytes);

    // pass 1: max|x| (bf16: packed maxima of the |x| bit patterns)
    uint32_t amax;
    if (BF16) {
      uint32_t m2 = 0;
      for (int64_t c = tt; c < nch; c += TT) {
        const uint4 v = buf[c];
        m2 = max_u16x2(max_u16x2(m2, v.x & 0x7fff7fffu),
                       max_u16x2(v.y & 0x7fff7fffu, max_u16x2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu)));
      }
      amax = max(m2 >> 16, m2 & 0xffffu) << 16;
    } else {
      float f = 0.0f;
      for (int64_t c = tt; c < nch; c += TT) {
        const uint4 v = buf[c];
        f = fmaxf(fmaxf(f, fabsf(__uint_as_float(v.x))),
                  fmaxf(fabsf(__uint_as_float(v.y)), fmaxf(fabsf(__uint_as_float(v.z)), fabsf(__uint_as_float(v.w)))));
      }
      amax = __float_as_uint(f);
    }
    amax = __reduce_max_sync(0xffffffffu, amax);
    if (T > 1) {
      if (lane == 0) red_max[warp] = amax;
      team_sync();
      for (int w = 0; w < T; ++w) amax = max(amax, red_max[team * T + w]);
    }
    float am = __uint_as_float(amax);
    if (am < kActClampEps) am = kActClampEps;
    const float sg = __fdiv_rn(127.0f, am);

    // pass 2: codes
    int8_t* qrow = a.xq + m * K;
    for (int64_t c = tt; c < nch; c += TT) {
      float x[kPer];
      unpack_chunk<BF16>(buf[c], x);
      uint32_t w[kPer / 4];
#pragma unroll
      for (int h = 0; h < kPer / 4; ++h)
        w[h] = pack_low_bytes(q8_bits(x[4 * h], sg), q8_bits(x[4 * h + 1], sg), q8_bits(x[4 * h + 2], sg),
                              q8_bits(x[4 * h + 3], sg));
      if (BF16) reinterpret_cast<uint2*>(qrow)[c] = make_uint2(w[0], w[1]);
      else reinterpret_cast<uint32_t*>(qrow)[c] = w[0];
    }
    if (leader) a.s[m] = sg;
    prev_st = st;
    if (++st == S) {
      st = 0;
      phase ^= 1u;
    }
  }
}

// Launch shape of the staged kernel, or ok = false where the one-CTA-per-row
// kernel serves (fewer than kRowStagedMinM rows, K % 16 != 0, or rows too
// long for a ring that keeps enough warps on each SM).
struct RowPlan {
  bool ok = false;
  int team = 1, warps = 0, stages = 0, grid = 0;
  size_t smem = 0;
};

constexpr int64_t kRowStagedMinM = 256;
constexpr size_t kRowSmemBudget = 200 * 1024;  // dynamic shared memory per CTA (also the kernel's limit)
constexpr int kRowWarpsPerSmTarget = 32;       // busy warps per SM the team size aims for
constexpr int kRowWarpsPerSmMin = 4;

template <bool BF16>
RowPlan plan_rows_staged(int64_t M, int64_t K, int num_sms) {
  RowPlan p;
  if (M < kRowStagedMinM || K % 16 != 0 || num_sms < 1) return p;
  const size_t row = (size_t)K * (BF16 ? 2 : 4);
  const size_t avail = kRowSmemBudget - kRowBarBytes;
  int S = row <= 4096 ? 4 : (row <= 8192 ? 3 : 2);
  // warps per row: several warps share a row (and its ring) when the rows are
  // too few, or the rings too large for the shared memory of an SM, to keep
  // about kRowWarpsPerSmTarget warps per SM at work
  const int64_t teams_per_sm = (int64_t)(228 * 1024) / ((int64_t)S * (int64_t)row + 1024);
  int T = 1;
  while (T < 8 && (M * T < (int64_t)kRowWarpsPerSmTarget * num_sms || teams_per_sm * T < kRowWarpsPerSmTarget))
    T *= 2;
  auto kern = quant_rows_staged_kernel<BF16>;
  if (set_smem_attrs(kern, kRowSmemBudget) != cudaSuccess) {
    (void)cudaGetLastError();  // not sticky: clear it so the fallback's launch check does not see it
    return p;
  }
  int nteams = 0, occ = 0, grid = 0;
  size_t smem = 0;
  for (int iter = 0; iter < 4; ++iter) {
    nteams = (int)std::min<size_t>(kRowWarpsMax / T, avail / ((size_t)S * row));
    if (nteams < 1) {
      if (S == 1) return p;
      --S;
      continue;
    }
    smem = kRowBarBytes + (size_t)nteams * S * row;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, nteams * T * 32, smem) != cudaSuccess) {
      (void)cudaGetLastError();
      return p;
    }
    if (occ < 1) return p;
    grid = (int)std::min<int64_t>((int64_t)num_sms * occ, (M + nteams - 1) / nteams);
    const int64_t rows_per_team = (M + (int64_t)grid * nteams - 1) / ((int64_t)grid * nteams);
    if (rows_per_team >= S || S == 1) break;
    S = (int)std::max<int64_t>(1, rows_per_team);  // no deeper ring than the rows a team gets
  }
  if (occ * nteams * T < kRowWarpsPerSmMin) return p;
  // the leader refills a stage at the top of the next row, after the team
  // barrier: with one stage that refill would come after the wait for the row
  // it carries, so a one-stage ring serves at most one row per team
  const int64_t rows_per_team = (M + (int64_t)grid * nteams - 1) / ((int64_t)grid * nteams);
  if (S == 1 && rows_per_team > 1) return p;
  p.ok = true;
  p.team = T;
  p.warps = nteams * T;
  p.stages = S;
  p.grid = grid;
  p.smem = smem;
  return p;
}

template <bool BF16>
cudaError_t launch_rows_staged(const void* X, int64_t M, int64_t K, int8_t* xq, float* s, int num_sms, uint32_t* err,
                               cudaStream_t stream, bool* launched, bool test_stall) {
  *launched = false;
  const RowPlan p = plan_rows_staged<BF16>(M, K, num_sms);
  if (!p.ok) return cudaSuccess;
  const RowQuantArgs a{static_cast<const char*>(X), M, K, xq, s, err, (uint32_t)(K * (BF16 ? 2 : 4)), p.stages, p.team,
                       test_stall ? 1 : 0};
  *launched = true;
  quant_rows_staged_kernel<BF16><<<p.grid, p.warps * 32, p.smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm_quant_act(const void* X, bool bf16, int64_t M, int64_t K, const float* gain, float eps,
                                     int8_t* xq, float* s, cudaStream_t stream) {
  // 128-bit path: every row starts 16-byte aligned, the gain vector too, and
  // each chunk's codes (8 or 4 bytes) are aligned stores
  const int esize = bf16 ? 2 : 4;
  const bool vec = (K * esize) % 16 == 0 && reinterpret_cast<uintptr_t>(X) % 16 == 0 &&
                   (!gain || reinterpret_cast<uintptr_t>(gain) % 16 == 0) &&
                   reinterpret_cast<uintptr_t>(xq) % (bf16 ? 8 : 4) == 0;
  const int64_t work = vec ? K * esize / 16 : K;
  int threads = (int)((work + 31) / 32 * 32);
  if (threads > 1024) threads = 1024;
  const unsigned long long rk = sq_recip((uint32_t)K);
  if (vec && rms_row_warps_serve(M, K * esize)) {
    const unsigned grid = (unsigned)((M + kRmsRowWarps - 1) / kRmsRowWarps);
    if (bf16)
      rmsnorm_quant_rows_kernel<true, 0><<<grid, 32 * kRmsRowWarps, 0, stream>>>(X, M, K, gain, eps, rk, xq, s,
                                                                                 nullptr, nullptr, 0);
    else
      rmsnorm_quant_rows_kernel<false, 0><<<grid, 32 * kRmsRowWarps, 0, stream>>>(X, M, K, gain, eps, rk, xq, s,
                                                                                  nullptr, nullptr, 0);
    return cudaGetLastError();
  }
  const X8Out none{};
  if (bf16)
    rmsnorm_quant_act_kernel<true, 0><<<(unsigned)M, threads, 0, stream>>>(X, K, vec, gain, eps, rk, xq, s, nullptr, none);
  else
    rmsnorm_quant_act_kernel<false, 0><<<(unsigned)M, threads, 0, stream>>>(X, K, vec, gain, eps, rk, xq, s, nullptr, none);
  return cudaGetLastError();
}

namespace {

// Threads of the RMS-norm kernels that write a GEMM operand: one 16-element
// group per thread in the codes pass, one 16-byte chunk per thread in the
// reductions.
int rmsnorm_operand_threads(int64_t K, bool bf16) {
  const int64_t chunks = K * (bf16 ? 2 : 4) / 16;
  int threads = (int)((chunks + 31) / 32 * 32);
  if (threads > 1024) threads = 1024;
  if (threads < 64) threads = 64;
  return threads;
}

}  // namespace

cudaError_t launch_rmsnorm_quant_act_x16(const void* X, bool bf16, int64_t M, int64_t K, const float* gain, float eps,
                                         int8_t* xq, float* s, void* x16, uint32_t* cnt, int ncnt,
                                         cudaStream_t stream) {
  const int threads = rmsnorm_operand_threads(K, bf16);
  const unsigned long long rk = sq_recip((uint32_t)K);
  X8Out counters{};
  counters.cnt = cnt;
  counters.ncnt = cnt ? ncnt : 0;
  uint4* o = static_cast<uint4*>(x16);
  if (rms_row_warps_serve(M, K * (bf16 ? 2 : 4))) {
    const unsigned grid = (unsigned)((M + kRmsRowWarps - 1) / kRmsRowWarps);
    if (bf16)
      rmsnorm_quant_rows_kernel<true, 1><<<grid, 32 * kRmsRowWarps, 0, stream>>>(X, M, K, gain, eps, rk, xq, s, o,
                                                                                 counters.cnt, counters.ncnt);
    else
      rmsnorm_quant_rows_kernel<false, 1><<<grid, 32 * kRmsRowWarps, 0, stream>>>(X, M, K, gain, eps, rk, xq, s, o,
                                                                                  counters.cnt, counters.ncnt);
    return cudaGetLastError();
  }
  if (bf16)
    rmsnorm_quant_act_kernel<true, 1><<<(unsigned)M, threads, 0, stream>>>(X, K, true, gain, eps, rk, xq, s, o, counters);
  else
    rmsnorm_quant_act_kernel<false, 1><<<(unsigned)M, threads, 0, stream>>>(X, K, true, gain, eps, rk, xq, s, o, counters);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_quant_act_x8(const void* X, bool bf16, int64_t M, int64_t K, const float* gain, float eps,
                                        int8_t* xq, float* s, void* ws, int num_sms, cudaStream_t stream) {
  const int threads = rmsnorm_operand_threads(K, bf16);
  const unsigned long long rk = sq_recip((uint32_t)K);
  const int BN = gemm_f8_token_tile(M);
  const X8Out o8{f8_operand(ws), f8_counters(ws, M, K, num_sms), num_sms, M, gemm_f8_kblocks(K), BN,
                 f8_sums(ws, M, K, num_sms)};
  const unsigned grid = (unsigned)((M + BN - 1) / BN * BN);  // every token of the last tile
  if (bf16)
    rmsnorm_quant_act_kernel<true, 2><<<grid, threads, 0, stream>>>(X, K, true, gain, eps, rk, xq, s, nullptr, o8);
  else
    rmsnorm_quant_act_kernel<false, 2><<<grid, threads, 0, stream>>>(X, K, true, gain, eps, rk, xq, s, nullptr, o8);
  return cudaGetLastError();
}

namespace {

// CTAs per token row for the fp8 operand writer: rows of at least 16384
// activations are split into slices of about 256 groups of 16 (at most 8, a
// portable cluster), while rows x CTAs stays within two waves of SMs.  Shorter
// rows, and the x_q-only quantisation, measured no faster split (the cluster
// launch costs about what the split saves there).
int row_split(int64_t rows, int64_t K, int num_sms) {
  if (K < 16384) return 1;
  int64_t S = (K / 16) / 256;
  if (S > 8) S = 8;
  while (S > 1 && rows * S > 2 * (int64_t)num_sms) --S;
  return S < 1 ? 1 : (int)S;
}

// quant_act_kernel over `rows` rows, each shared by a cluster of S CTAs.
template <bool BF16, int OUT>
cudaError_t launch_rows(int64_t rows, int S, int threads, cudaStream_t stream, const void* X, int64_t K, bool vec,
                        int8_t* xq, float* s, uint4* xop, const X8Out& o8) {
  if (S <= 1) {
    quant_act_kernel<BF16, OUT><<<(unsigned)rows, threads, 0, stream>>>(X, K, vec, xq, s, xop, o8);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * S));
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_act_kernel<BF16, OUT>, X, K, vec, xq, s, xop, o8);
}

int threads_for(int64_t work) {
  int threads = (int)((work + 31) / 32 * 32);
  if (threads > 1024) threads = 1024;
  if (threads < 64) threads = 64;
  return threads;
}

}  // namespace

cudaError_t launch_quant_act(const void* X, bool bf16, int64_t M, int64_t K, int8_t* xq, float* s, int num_sms,
                             uint32_t* err, cudaStream_t stream, bool test_stall) {
  if (reinterpret_cast<uintptr_t>(X) % 16 == 0 && reinterpret_cast<uintptr_t>(xq) % 16 == 0) {
    bool launched = false;
    const cudaError_t e = bf16 ? launch_rows_staged<true>(X, M, K, xq, s, num_sms, err, stream, &launched, test_stall)
                               : launch_rows_staged<false>(X, M, K, xq, s, num_sms, err, stream, &launched, test_stall);
    if (e != cudaSuccess || launched) return e;
  }
  const int esize = bf16 ? 2 : 4;
  const bool vec = (K * esize) % 16 == 0;
  const int64_t work = vec ? K * esize / 16 : K;
  const int S = 1;  // one CTA per row (see row_split)
  const int threads = threads_for((work + S - 1) / S);
  const X8Out none{};
  return bf16 ? launch_rows<true, 0>(M, S, threads, stream, X, K, vec, xq, s, nullptr, none)
              : launch_rows<false, 0>(M, S, threads, stream, X, K, vec, xq, s, nullptr, none);
}

cudaError_t launch_quant_act_x16(const void* X, bool bf16, int64_t M, int64_t K, int8_t* xq, float* s, void* x16,
                                 uint32_t* cnt, int ncnt, cudaStream_t stream) {
  // one 16-element group per thread in the second pass (K % 16 == 0)
  int threads = (int)((K / 16 + 31) / 32 * 32);
  if (threads > 1024) threads = 1024;
  if (threads < 64) threads = 64;
  uint4* o = static_cast<uint4*>(x16);
  X8Out counters{};
  counters.cnt = cnt;
  counters.ncnt = cnt ? ncnt : 0;
  if (bf16) quant_act_kernel<true, 1><<<(unsigned)M, threads, 0, stream>>>(X, K, true, xq, s, o, counters);
  else quant_act_kernel<false, 1><<<(unsigned)M, threads, 0, stream>>>(X, K, true, xq, s, o, counters);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_x8(const void* X, bool bf16, int64_t M, int64_t K, int8_t* xq, float* s, void* ws,
                                int num_sms, cudaStream_t stream) {
  const int BN = gemm_f8_token_tile(M);
  const X8Out o8{f8_operand(ws), f8_counters(ws, M, K, num_sms), num_sms, M, gemm_f8_kblocks(K), BN,
                 f8_sums(ws, M, K, num_sms)};
  const int64_t rows = (M + BN - 1) / BN * BN;  // every token of the last tile
  const int S = row_split(rows, K, num_sms);
  const int threads = threads_for((K / 16 + S - 1) / S);
  return bf16 ? launch_rows<true, 2>(rows, S, threads, stream, X, K, true, xq, s, nullptr, o8)
              : launch_rows<false, 2>(rows, S, threads, stream, X, K, true, xq, s, nullptr, o8);
}

}  // namespace bl
