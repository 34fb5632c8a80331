// pack.cu -- absmean ternarisation and 2-bit packing of a latent weight matrix.
//
// gamma = mean|W| (absmean quantiser: anthology note-168 on arXiv 2402.17764,
// "What it does"; yousumm.com BitNet b1.58 2B4T transcript, "ABS mean
// quantizer" paragraph) is computed EXACTLY, so it does not depend on the
// order in which thousands of threads add their values:
//
//   |w| = m * 2^(e-150) for the 24-bit significand m and biased exponent e
//   (subnormals: e := 1, no hidden bit).  Split e into a group g = e >> 3 and
//   an offset e & 7; then m << (e & 7) < 2^31 and
//       sum|w| = sum_g B[g] * 2^(8g - 150),  B[g] = sum over group g of (m << (e & 7)).
//   Each B[g] is an integer sum, so it is the same in any order.  A thread
//   keeps two register sums for the two highest groups it has seen (a
//   Gaussian matrix spends >99% of its values there) and sends the rest to
//   shared-memory buckets; CTAs add their buckets into 32 global u64 buckets.
//   One thread then forms the 312-bit total, divides by N*K and rounds once to
//   fp32 (round half to even).
//
// Ternarisation W_q = clip(rint(W / d), -1, 1) with d = fp32(gamma + eps)
// needs no division per weight: IEEE division rounds monotonically, so
// fl(|w|/d) <= 1/2 exactly when the real quotient |w|/d <= 1/2 + 2^-25 (the
// midpoint between 0.5 and the next fp32, which rounds to the even 0.5), and
// rint maps every value <= 1/2 to 0 and every larger one to +-1 after the
// clip.  d*(1/2 + 2^-25) has at most 49 significant bits, so it is exact in
// fp64; rounding it down to fp32 gives a threshold T with |w| <= T exactly
// when W_q = 0.  For non-negative floats, comparing bit patterns compares
// values, so each weight costs one integer compare.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace bl {
namespace {

struct AbsmeanAcc {
  uint32_t G = 0;              // current highest group of this thread
  unsigned long long hi = 0;   // sum for group G
  unsigned long long lo = 0;   // sum for group G - 1
  uint32_t nonfinite = 0;

  __device__ __forceinline__ void add(float w, unsigned long long* sb) {
    const uint32_t u = __float_as_uint(w) & 0x7fffffffu;
    const uint32_t e = u >> 23;
    if (e == 255u) {
      nonfinite = 1;
      return;
    }
    uint32_t m = u & 0x7fffffu;
    uint32_t ee = e;
    if (e) m |= 0x800000u;
    else ee = 1u;
    const uint32_t g = ee >> 3;
    const uint32_t v = m << (ee & 7u);
    if (g == G) {
      hi += v;
    } else if (g + 1u == G) {
      lo += v;
    } else if (g > G) {
      if (g == G + 1u) {
        if (G >= 1u && lo) atomicAdd(&sb[G - 1u], lo);
        lo = hi;
      } else {
        if (hi) atomicAdd(&sb[G], hi);
        if (G >= 1u && lo) atomicAdd(&sb[G - 1u], lo);
        lo = 0;
      }
      hi = v;
      G = g;
    } else {
      atomicAdd(&sb[g], (unsigned long long)v);
    }
  }

  __device__ __forceinline__ void add4(const float4& v, unsigned long long* sb) {
    add(v.x, sb);
    add(v.y, sb);
    add(v.z, sb);
    add(v.w, sb);
  }

  __device__ __forceinline__ void flush(unsigned long long* sb) {
    if (hi) atomicAdd(&sb[G], hi);
    if (G >= 1u && lo) atomicAdd(&sb[G - 1u], lo);
  }

  // Warp-wide flush: where every lane holds the same top group G (the common
  // case: a weight matrix's magnitudes span a few binades), the register sums
  // are added across the warp first and one lane issues the two atomics, so a
  // CTA's threads do not serialise on the same two shared buckets.  Integer
  // sums, so the result is the same in any order.  All 32 lanes must call it.
  __device__ __forceinline__ void flush_warp(unsigned long long* sb) {
    int same = 0;
    __match_all_sync(0xffffffffu, G, &same);
    if (!same) {
      flush(sb);
      return;
    }
    unsigned long long h = hi, l = lo;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      h += __shfl_xor_sync(0xffffffffu, h, off);
      l += __shfl_xor_sync(0xffffffffu, l, off);
    }
    if ((threadIdx.x & 31u) == 0) {
      if (h) atomicAdd(&sb[G], h);
      if (G >= 1u && l) atomicAdd(&sb[G - 1u], l);
    }
  }
};

constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kPackThreads) absmean_hist_kernel(const float4* __restrict__ W4, uint64_t n4,
                                                                     PackWorkspace* __restrict__ ws) {
  __shared__ unsigned long long sb[32];
  __shared__ uint32_t snf;
  if (threadIdx.x < 32) sb[threadIdx.x] = 0;
  if (threadIdx.x == 0) snf = 0;
  __syncthreads();

  AbsmeanAcc acc;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(W4 + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) acc.add4(v[u], sb);
  }
  for (; i < n4; i += stride) acc.add4(__ldg(W4 + i), sb);
  acc.flush_warp(sb);
  if (acc.nonfinite) snf = 1;
  __syncthreads();
  if (threadIdx.x < 32 && sb[threadIdx.x]) atomicAdd(&ws->bucket[threadIdx.x], sb[threadIdx.x]);
  if (threadIdx.x == 0 && snf) atomicOr(&ws->nonfinite, 1u);
}

// Bit i of a little-endian array of 32-bit limbs.
__device__ __forceinline__ uint32_t limb_bit(const uint32_t* q, int i) { return (q[i >> 5] >> (i & 31)) & 1u; }

__global__ void absmean_finish_kernel(PackWorkspace* __restrict__ ws, uint64_t n, float eps, float* __restrict__ gamma) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  constexpr int L = 12;  // 384-bit total: sum < 2^(8*31 + 63)
  float g;
  if (ws->nonfinite) {
    g = __int_as_float(0x7fc00000);
  } else {
    uint32_t S[L];
    for (int i = 0; i < L; ++i) S[i] = 0;
    for (int b = 0; b < 32; ++b) {
      const unsigned long long B = ws->bucket[b];
      if (!B) continue;
      const int li = b >> 2, sh = 8 * (b & 3);
      const unsigned long long low = B << sh;
      const uint32_t part[3] = {(uint32_t)low, (uint32_t)(low >> 32), sh ? (uint32_t)(B >> (64 - sh)) : 0u};
      unsigned long long carry = 0;
      for (int i = li; i < L; ++i) {
        const unsigned long long t = (unsigned long long)S[i] + (i - li < 3 ? part[i - li] : 0u) + carry;
        S[i] = (uint32_t)t;
        carry = t >> 32;
        if (i - li >= 2 && !carry) break;
      }
    }
    // Q = floor(S / n), R = S mod n  (n <= 2^32, so the running remainder fits 64 bits)
    uint32_t Q[L];
    unsigned long long R = 0;
    for (int i = L - 1; i >= 0; --i) {
      const unsigned long long cur = (R << 32) | S[i];
      Q[i] = (uint32_t)(cur / n);
      R = cur % n;
    }
    // mean = (Q + R/n) * 2^-150.  Keep 24 bits from the top set bit down, but no
    // finer than the subnormal quantum 2^-149 (= 2 units).
    int p = -1;
    for (int i = L - 1; i >= 0 && p < 0; --i)
      if (Q[i]) p = i * 32 + (31 - __clz(Q[i]));
    int qe = p - 23 > 1 ? p - 23 : 1;
    uint32_t mant = 0;
    for (int b = p; b >= qe; --b) mant = (mant << 1) | limb_bit(Q, b);
    const uint32_t round_bit = limb_bit(Q, qe - 1);
    bool sticky = R != 0;
    for (int b = 0; b < qe - 1 && !sticky; ++b) sticky = limb_bit(Q, b) != 0;
    if (round_bit && (sticky || (mant & 1u))) {
      ++mant;
      if (mant == (1u << 24)) {
        mant = 1u << 23;
        ++qe;
      }
    }
    uint32_t bits;
    if (mant >= (1u << 23)) bits = qe >= 255 ? 0x7f800000u : (((uint32_t)qe << 23) | (mant - (1u << 23)));
    else bits = mant;  // subnormal (qe == 1): mant * 2^-149
    g = __uint_as_float(bits);
  }
  *gamma = g;
  const float d = __fadd_rn(g, eps);
  const double thr = (double)d * (0.5 + 0x1p-25);  // exact
  ws->gamma = g;
  ws->thresh_bits = __float_as_uint(__double2float_rd(thr));
}

__device__ __forceinline__ uint32_t ternary_code(float w, uint32_t T) {
  const uint32_t u = __float_as_uint(w);
  return (u & 0x7fffffffu) <= T ? 1u : ((u >> 31) ? 0u : 2u);
}

__global__ void __launch_bounds__(kPackThreads) ternarize_pack_kernel(const float4* __restrict__ W4, uint64_t n4,
                                                                       const PackWorkspace* __restrict__ ws,
                                                                       uint8_t* __restrict__ Wp) {
  const uint32_t T = ws->thresh_bits;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcs(W4 + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      Wp[i + u * stride] = (uint8_t)(ternary_code(v[u].x, T) | (ternary_code(v[u].y, T) << 2) |
                                     (ternary_code(v[u].z, T) << 4) | (ternary_code(v[u].w, T) << 6));
  }
  for (; i < n4; i += stride) {
    const float4 v = __ldcs(W4 + i);
    Wp[i] = (uint8_t)(ternary_code(v.x, T) | (ternary_code(v.y, T) << 2) | (ternary_code(v.z, T) << 4) |
                      (ternary_code(v.w, T) << 6));
  }
}

// Base-3 packing, five weights per byte: byte j of row n is the sum over
// i < 5 of code(W[n, 5j + i]) * 3^i, with the code of the 2-bit format (q + 1,
// the same zero band); positions at or past K count as code 1 (q = 0), so a
// padding byte is 121.  One thread per output byte; a warp's five loads fall
// on the same 640 contiguous bytes of W, so the last four hit L1.
__global__ void __launch_bounds__(kPackThreads) ternarize_pack_tq5_kernel(const float* __restrict__ W, int64_t N,
                                                                           int64_t K, int64_t pitch,
                                                                           const PackWorkspace* __restrict__ ws,
                                                                           uint8_t* __restrict__ Wt) {
  const uint32_t T = ws->thresh_bits;
  const int64_t total = N * pitch;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = idx / pitch, j = idx - n * pitch;
    const float* row = W + n * K;
    uint32_t v = 0, w = 1;
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      const int64_t k = 5 * j + i;
      v += (k < K ? ternary_code(__ldg(row + k), T) : 1u) * w;
      w *= 3u;
    }
    Wt[idx] = (uint8_t)v;
  }
}

}  // namespace

cudaError_t launch_pack_tq5(const float* W, int64_t N, int64_t K, int64_t pitch, float eps, uint8_t* Wt,
                            float* gamma, PackWorkspace* ws, int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(PackWorkspace), stream);
  if (e != cudaSuccess) return e;
  const uint64_t n = (uint64_t)N * (uint64_t)K, n4 = n / 4;
  const uint64_t want = (n4 + kPackThreads - 1) / kPackThreads;
  const int grid = (int)(want < (uint64_t)num_sms * 8 ? (want ? want : 1) : (uint64_t)num_sms * 8);
  absmean_hist_kernel<<<grid, kPackThreads, 0, stream>>>(reinterpret_cast<const float4*>(W), n4, ws);
  absmean_finish_kernel<<<1, 32, 0, stream>>>(ws, n, eps, gamma);
  const uint64_t bytes = (uint64_t)N * (uint64_t)pitch;
  const uint64_t want2 = (bytes + kPackThreads - 1) / kPackThreads;
  const int grid2 = (int)(want2 < (uint64_t)num_sms * 16 ? want2 : (uint64_t)num_sms * 16);
  ternarize_pack_tq5_kernel<<<grid2, kPackThreads, 0, stream>>>(W, N, K, pitch, ws, Wt);
  return cudaGetLastError();
}

cudaError_t launch_pack(const float* W, uint64_t n, float eps, uint8_t* Wp, float* gamma, PackWorkspace* ws,
                        int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(PackWorkspace), stream);
  if (e != cudaSuccess) return e;
  const uint64_t n4 = n / 4;
  const uint64_t want = (n4 + kPackThreads - 1) / kPackThreads;
  const int grid = (int)(want < (uint64_t)num_sms * 8 ? (want ? want : 1) : (uint64_t)num_sms * 8);
  absmean_hist_kernel<<<grid, kPackThreads, 0, stream>>>(reinterpret_cast<const float4*>(W), n4, ws);
  absmean_finish_kernel<<<1, 32, 0, stream>>>(ws, n, eps, gamma);
  ternarize_pack_kernel<<<grid, kPackThreads, 0, stream>>>(reinterpret_cast<const float4*>(W), n4, ws, Wp);
  return cudaGetLastError();
}

}  // namespace bl
