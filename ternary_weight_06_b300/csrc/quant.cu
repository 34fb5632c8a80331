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
#include <cstdint>

#include "common.cuh"
#include "internal.h"

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

template <bool BF16, bool X16>
__global__ void __launch_bounds__(1024) quant_act_kernel(const void* __restrict__ X, int64_t K, bool vec,
                                                         int8_t* __restrict__ xq, float* __restrict__ s,
                                                         uint4* __restrict__ x16) {
  constexpr int kEsize = BF16 ? 2 : 4;
  const int64_t m = blockIdx.x;
  const char* row = static_cast<const char*>(X) + m * K * kEsize;
  int8_t* out = xq + m * K;
  const int tid = threadIdx.x, nt = blockDim.x;

  uint32_t amax = 0;
  if (vec) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int64_t nch = K * kEsize / 16;
    for (int64_t c = tid; c < nch; c += nt) {
      const uint4 v = __ldg(r4 + c);
      if (BF16) {
        amax = max(amax, max(max(abs_bits_bf16x2(v.x), abs_bits_bf16x2(v.y)),
                             max(abs_bits_bf16x2(v.z), abs_bits_bf16x2(v.w))));
      } else {
        amax = max(amax, max(max(v.x & 0x7fffffffu, v.y & 0x7fffffffu), max(v.z & 0x7fffffffu, v.w & 0x7fffffffu)));
      }
    }
  } else {
    for (int64_t k = tid; k < K; k += nt) {
      uint32_t b = BF16 ? ((uint32_t)reinterpret_cast<const uint16_t*>(row)[k] << 16)
                        : reinterpret_cast<const uint32_t*>(row)[k];
      amax = max(amax, b & 0x7fffffffu);
    }
  }
  __shared__ uint32_t red[32];
  amax = __reduce_max_sync(0xffffffffu, amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid < 32) {
    uint32_t v = tid < (nt >> 5) ? red[tid] : 0u;
    v = __reduce_max_sync(0xffffffffu, v);
    if (tid == 0) red[0] = v;
  }
  __syncthreads();
  float a = __uint_as_float(red[0]);
  if (a < kActClampEps) a = kActClampEps;
  const float sm = __fdiv_rn(127.0f, a);
  if (tid == 0) s[m] = sm;

  if (X16) {
    // groups of 16 activations: x_q (natural order) and the GEMM's fp16 operand
    // (order p = 4i + j within the group); K % 16 == 0
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    uint4* xo = x16 + m * (K / 8);
    for (int64_t g = tid; g < K / 16; g += nt) {
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
      uint32_t h[8];
      convert_x16_f16(q4, h);
      xo[2 * g] = make_uint4(h[0], h[1], h[2], h[3]);
      xo[2 * g + 1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  } else if (vec) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int64_t nch = K * kEsize / 16;
    for (int64_t c = tid; c < nch; c += nt) {
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
    for (int64_t k = tid; k < K; k += nt) {
      const float x = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(row)[k] << 16)
                           : reinterpret_cast<const float*>(row)[k];
      out[k] = (int8_t)q8(x, sm);
    }
  }
}

// Sub-layer RMS normalisation folded into the quantisation.  The RMS factor
// 1/sqrt(mean(x^2) + eps) is one positive number per token, to which absmax
// codes are invariant, so the codes are those of x * gain and only the scale
// changes: s = s(x * gain) * sqrt(mean(x^2) + eps).  Pass 1 forms max|x * g|
// (order-free, on bit patterns) and sum x^2 (fp64); pass 2 quantises x * g
// with the same fp32 product, so x_q is bit-identical to quantising x * g.
template <bool BF16>
__global__ void __launch_bounds__(1024) rmsnorm_quant_act_kernel(const void* __restrict__ X, int64_t K,
                                                                 const float* __restrict__ gain, float eps,
                                                                 int8_t* __restrict__ xq, float* __restrict__ s) {
  constexpr int kEsize = BF16 ? 2 : 4;
  const int64_t m = blockIdx.x;
  const char* row = static_cast<const char*>(X) + m * K * kEsize;
  int8_t* out = xq + m * K;
  const int tid = threadIdx.x, nt = blockDim.x;
  auto load = [&](int64_t k) -> float {
    return BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(row)[k] << 16)
                : reinterpret_cast<const float*>(row)[k];
  };
  uint32_t amax = 0;
  double ss = 0.0;
  for (int64_t k = tid; k < K; k += nt) {
    const float x = load(k);
    const float xg = gain ? __fmul_rn(x, __ldg(gain + k)) : x;
    amax = max(amax, __float_as_uint(xg) & 0x7fffffffu);
    ss = __fma_rn((double)x, (double)x, ss);
  }
  __shared__ uint32_t red[32];
  __shared__ double red_ss[32];
  amax = __reduce_max_sync(0xffffffffu, amax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) {
    red[tid >> 5] = amax;
    red_ss[tid >> 5] = ss;
  }
  __syncthreads();
  if (tid < 32) {
    uint32_t v = tid < (nt >> 5) ? red[tid] : 0u;
    double w = tid < (nt >> 5) ? red_ss[tid] : 0.0;
    v = __reduce_max_sync(0xffffffffu, v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (tid == 0) {
      red[0] = v;
      red_ss[0] = w;
    }
  }
  __syncthreads();
  float a = __uint_as_float(red[0]);
  if (a < kActClampEps) a = kActClampEps;
  const float sg = __fdiv_rn(127.0f, a);
  if (tid == 0) s[m] = (float)((double)sg * sqrt(red_ss[0] / (double)K + (double)eps));
  for (int64_t k = tid; k < K; k += nt) {
    const float x = load(k);
    const float xg = gain ? __fmul_rn(x, __ldg(gain + k)) : x;
    out[k] = (int8_t)q8(xg, sg);
  }
}

}  // namespace

cudaError_t launch_rmsnorm_quant_act(const void* X, bool bf16, int64_t M, int64_t K, const float* gain, float eps,
                                     int8_t* xq, float* s, cudaStream_t stream) {
  int threads = (int)((K + 31) / 32 * 32);
  if (threads > 1024) threads = 1024;
  if (bf16) rmsnorm_quant_act_kernel<true><<<(unsigned)M, threads, 0, stream>>>(X, K, gain, eps, xq, s);
  else rmsnorm_quant_act_kernel<false><<<(unsigned)M, threads, 0, stream>>>(X, K, gain, eps, xq, s);
  return cudaGetLastError();
}

cudaError_t launch_quant_act(const void* X, bool bf16, int64_t M, int64_t K, int8_t* xq, float* s,
                             cudaStream_t stream) {
  const int esize = bf16 ? 2 : 4;
  const bool vec = (K * esize) % 16 == 0;
  const int64_t work = vec ? K * esize / 16 : K;
  int threads = (int)((work + 31) / 32 * 32);
  if (threads > 1024) threads = 1024;
  if (threads < 32) threads = 32;
  if (bf16) quant_act_kernel<true, false><<<(unsigned)M, threads, 0, stream>>>(X, K, vec, xq, s, nullptr);
  else quant_act_kernel<false, false><<<(unsigned)M, threads, 0, stream>>>(X, K, vec, xq, s, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_x16(const void* X, bool bf16, int64_t M, int64_t K, int8_t* xq, float* s, void* x16,
                                 cudaStream_t stream) {
  // one 16-element group per thread in the second pass (K % 16 == 0)
  int threads = (int)((K / 16 + 31) / 32 * 32);
  if (threads > 1024) threads = 1024;
  if (threads < 64) threads = 64;
  uint4* o = static_cast<uint4*>(x16);
  if (bf16) quant_act_kernel<true, true><<<(unsigned)M, threads, 0, stream>>>(X, K, true, xq, s, o);
  else quant_act_kernel<false, true><<<(unsigned)M, threads, 0, stream>>>(X, K, true, xq, s, o);
  return cudaGetLastError();
}

}  // namespace bl
