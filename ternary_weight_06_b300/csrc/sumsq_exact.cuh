// sumsq_exact.cuh -- the exact sum of squares of a row of fp32 values, and
// its mean rounded once to fp32, for the sub-layer RMS normalisation.
//
// mean(x^2) is taken as the exact real mean of the squares, rounded once to
// fp32 (ties to even), so it does not depend on the order in which threads
// add their values.  With x = sig * 2^(ee - 150) (24-bit significand sig,
// biased exponent ee, ee := 1 for subnormals), x^2 = sig^2 * 2^(2 ee - 300).
// Split ee into a group g = ee >> 3 and an offset ee & 7:
//     x^2 = (sig^2 << 2 (ee & 7)) * 2^(16 g - 300),  sig^2 << 2 (ee & 7) < 2^62,
// so a 128-bit integer per group holds the exact sum of up to 2^66 squares,
// and the total is sum_g B[g] * 2^(16 g) units of 2^-300 (below 2^582 for
// rows of up to 2^24 values).  With the row's top group known (from max|x|),
// a thread keeps 128-bit register sums for it and the group below (an
// activation row spends almost all of its values there) and adds the others
// into 32 shared 128-bit buckets; one warp then forms the total, divides it
// by K exactly and rounds once.
#pragma once

#include <cstdint>

namespace bl {

constexpr int kSqGroups = 32;

// 32 exact 128-bit sums (hi:lo) in shared memory.
struct SqBuckets {
  unsigned long long lo[kSqGroups];
  unsigned long long hi[kSqGroups];
};

__device__ __forceinline__ void sq_clear(SqBuckets* sb) {
  for (int i = threadIdx.x; i < kSqGroups; i += blockDim.x) {
    sb->lo[i] = 0;
    sb->hi[i] = 0;
  }
}

// Adds the 128-bit value (v1:v0) into bucket g.  The carry out of the low
// word is taken from the atomic's own old value, so concurrent adds stay
// exact in any order.
__device__ __forceinline__ void sq_bucket_add(SqBuckets* sb, uint32_t g, unsigned long long v0,
                                              unsigned long long v1) {
  if (v0) {
    const unsigned long long old = atomicAdd(&sb->lo[g], v0);
    v1 += (old + v0 < old) ? 1ull : 0ull;
  }
  if (v1) atomicAdd(&sb->hi[g], v1);
}

// Per-thread sums for a row whose top group G (that of max|x|) is known:
// every value's group is <= G, groups G and G - 1 (nearly all values of an
// activation row) are summed in registers, any other value is added to its
// shared bucket directly.
struct SqAcc {
  uint32_t G;
  unsigned long long h0 = 0, h1 = 0;  // group G
  unsigned long long l0 = 0, l1 = 0;  // group G - 1

  __device__ __forceinline__ explicit SqAcc(uint32_t top_group) : G(top_group) {}

  __device__ __forceinline__ static void add128(unsigned long long& a0, unsigned long long& a1,
                                                unsigned long long v) {
    a0 += v;
    a1 += (a0 < v) ? 1ull : 0ull;
  }

  // x finite (a non-finite x gives an unspecified sum, never a fault).
  __device__ __forceinline__ void add(float x, SqBuckets* sb) {
    const uint32_t u = __float_as_uint(x) & 0x7fffffffu;
    if (u == 0) return;
    const uint32_t e = u >> 23;
    const uint32_t sig = (u & 0x7fffffu) | (e ? 0x800000u : 0u);
    const uint32_t ee = e ? e : 1u;
    const uint32_t g = (ee >> 3) & (kSqGroups - 1);
    const unsigned long long v = ((unsigned long long)sig * sig) << (2u * (ee & 7u));
    if (g == G) add128(h0, h1, v);
    else if (g + 1u == G) add128(l0, l1, v);
    else sq_bucket_add(sb, g, v, 0);
  }

  // Every lane of the warp must call it (all share G): the register sums are
  // added across the warp (128-bit adds with carry) and one lane adds them to
  // the buckets, so the warps of a CTA do not serialise on the same buckets.
  __device__ __forceinline__ void flush_warp(SqBuckets* sb) {
    unsigned long long a0 = h0, a1 = h1, b0 = l0, b1 = l1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long ra0 = __shfl_xor_sync(0xffffffffu, a0, off);
      const unsigned long long ra1 = __shfl_xor_sync(0xffffffffu, a1, off);
      const unsigned long long rb0 = __shfl_xor_sync(0xffffffffu, b0, off);
      const unsigned long long rb1 = __shfl_xor_sync(0xffffffffu, b1, off);
      a0 += ra0;
      a1 += ra1 + ((a0 < ra0) ? 1ull : 0ull);
      b0 += rb0;
      b1 += rb1 + ((b0 < rb0) ? 1ull : 0ull);
    }
    if ((threadIdx.x & 31u) == 0) {
      sq_bucket_add(sb, G, a0, a1);
      if (G >= 1u) sq_bucket_add(sb, G - 1u, b0, b1);
    }
  }
};

// Group of a finite value's squares (see above): that of max|x| bounds them all.
__device__ __forceinline__ uint32_t sq_group(uint32_t abs_bits) {
  const uint32_t e = abs_bits >> 23;
  return ((e ? e : 1u) >> 3) & (kSqGroups - 1);
}

// floor((2^64 - 1) / K): the reciprocal sq_mean_f32 divides with (host side).
inline unsigned long long sq_recip(uint32_t K) { return 0xffffffffffffffffull / K; }

// mean = (sum_g B[g] * 2^(16 g)) / K units of 2^-300, rounded once to fp32
// (ties to even; +inf above the fp32 range).  1 <= K <= 2^24, recip =
// sq_recip(K).  Called by all 32 lanes of one warp; every lane returns the
// result.  Lane i (< 20) holds 32-bit word i of the 640-bit numbers, so no
// array is indexed at run time and everything stays in registers; the loops
// stay rolled (small code: the finish runs once per row):
//   1. lane i adds up the parts of the (at most 12) groups that overlap its
//      word, in 64 bits (12 parts of < 2^32 each);
//   2. the carries run from word 0 up, 20 uniform shuffle steps;
//   3. the division by K runs from word 19 down, 20 uniform steps; each
//      divides cur = R * 2^32 + S[i] < 2^56 with the reciprocal (the estimate
//      is q or q - 1: the reciprocal is off by less than 2 and cur * 2 <
//      2^57), and one correction makes it exact;
//   4. rounding: 24 bits from the top set bit p down, but no finer than the
//      subnormal quantum 2^-149 = 2^151 units; round bit and sticky bit from
//      the bits below, and the remainder.
__device__ __noinline__ float sq_mean_f32(const SqBuckets* sb, uint32_t K, unsigned long long recip) {
  constexpr unsigned kFull = 0xffffffffu;
  constexpr int kWords = 20;   // 640 bits
  constexpr int kQmin = 151;   // bit index of the subnormal quantum
  const int lane = (int)(threadIdx.x & 31u);
  unsigned long long v = 0;
  if (lane < kWords) {
#pragma unroll 1
    for (int j = 0; j < 12; ++j) {
      const int g = 2 * (lane - 5) + j;  // groups whose 144 shifted bits overlap word `lane`
      if (g >= 0 && g < kSqGroups) {
        const unsigned long long lo = sb->lo[g], hi = sb->hi[g];
        const int sh = 16 * (g & 1);
        const int pi = lane - (g >> 1);  // 32-bit part of the shifted bucket, 0..5
        unsigned long long w;
        if (pi < 2) w = lo << sh;
        else if (pi < 4) w = sh ? ((lo >> (64 - sh)) | (hi << sh)) : hi;
        else w = sh ? (hi >> (64 - sh)) : 0ull;
        v += (pi & 1) ? (w >> 32) : (w & 0xffffffffull);
      }
    }
  }
  uint32_t S = 0;
  unsigned long long carry = 0;
#pragma unroll 1
  for (int i = 0; i < kWords; ++i) {
    const unsigned long long t = __shfl_sync(kFull, v, i) + carry;
    if (lane == i) S = (uint32_t)t;
    carry = t >> 32;
  }
  uint32_t Q = 0;
  unsigned long long R = 0;
#pragma unroll 1
  for (int i = kWords - 1; i >= 0; --i) {
    const unsigned long long cur = (R << 32) | __shfl_sync(kFull, S, i);
    unsigned long long q = __umul64hi(cur, recip);
    unsigned long long r = cur - q * K;
    if (r >= K) {
      r -= K;
      ++q;
    }
    if (lane == i) Q = (uint32_t)q;
    R = r;
  }
  const int p = __reduce_max_sync(kFull, Q ? lane * 32 + 31 - (int)__clz(Q) : -1);
  int qe = p - 23 > kQmin ? p - 23 : kQmin;
  const int w0 = qe >> 5;  // <= 19 (p <= 639)
  const unsigned long long win = (((unsigned long long)__shfl_sync(kFull, Q, (w0 + 1) & 31) << 32) |
                                  __shfl_sync(kFull, Q, w0)) >> (qe & 31);
  uint32_t mant = p >= qe ? (uint32_t)win & ((1u << (p - qe + 1)) - 1u) : 0u;
  const int rb = qe - 1, wr = rb >> 5;
  const uint32_t round_bit = (__shfl_sync(kFull, Q, wr) >> (rb & 31)) & 1u;
  const uint32_t below = lane < wr ? Q : (lane == wr ? (Q & ((1u << (rb & 31)) - 1u)) : 0u);
  const bool sticky = R != 0 || __any_sync(kFull, below != 0);
  if (round_bit && (sticky || (mant & 1u))) {
    ++mant;
    if (mant == (1u << 24)) {
      mant = 1u << 23;
      ++qe;
    }
  }
  uint32_t bits;
  if (mant >= (1u << 23)) {
    const int biased = qe - 150;  // value = mant * 2^(qe - 300), mant in [2^23, 2^24)
    bits = biased >= 255 ? 0x7f800000u : (((uint32_t)biased << 23) | (mant - (1u << 23)));
  } else {
    bits = mant;  // subnormal (qe == kQmin): mant * 2^-149
  }
  return __uint_as_float(bits);
}

}  // namespace bl
