// gemv_lut.cu -- the ternary GEMV by table lookup, the approach of the CPU
// kernels the BitNet b1.58 pages point to (promptinjection.net, "4. GPU
// Support: The Fragile Boost": GPU inference still rests on lookup tables),
// built here as a comparison variant of the conditional-add GEMV.
//
// For every pair of activations (x[2p], x[2p+1]) of a token, a 16-entry table
// holds sum_i (c_i - 1) x[2p+i] for every 4-bit value c0 + 4 c1 of two packed
// codes.  A packed byte holds two such nibbles, so the product becomes one
// table lookup and one integer add per two weights:
//     acc[n] = sum_p T_p[nibble p of row n]
// exact in int32 (every entry is an integer of magnitude <= 256, int16).
//
// Tables live in shared memory, a K-slice of up to 8192 activations at a time
// (128 KB); each CTA owns a contiguous block of output rows, builds the
// tables of the current token and slice, then its 16 warps stream their rows
// (warp w takes rows w, w + 16, ...): lane l of a warp loads 16-byte words
// l, l + 32, l + 64, l + 96 of the row's slice, the next row's words already
// in flight while it looks up the current row's 32 nibbles per word.  The
// table is laid out so that, for any codes, the 32 lanes of a lookup (same i
// and u, v = lane + 32 j) touch 32 different banks, and so that an entry's
// byte offset is the nibble shifted into place or-ed with a per-lane base:
//     entry (nib, i, u, v) at byte nib * 8192 + i * 1024 + (u >> 1) * 512
//                                  + 4 v + 2 (u & 1)
// for pair p = 8 w + i of 32-bit word w = 4 v + u of the slice (the entries
// of u = 2 h and 2 h + 1 share a 32-bit word).  Row sums are
// reduced across the warp and kept per CTA; the epilogue is that of every
// forward kernel: y = fp32(fp32(acc) * fp32(gamma / s[m])).
// The weights are read once per token.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace bl {
namespace {

constexpr int kLutThreads = 512;
constexpr int kLutWarps = kLutThreads / 32;
constexpr int kSliceK = 8192;              // activations per table slice
constexpr int kL4 = kSliceK / 64;          // 16-byte words of packed weights per row and slice
constexpr int kWordsPerLane = kL4 / 32;    // 4
constexpr int kTableBytes = 16 * 8 * 4 * kL4 * 2;  // 128 KB of int16 entries

struct LutCfg {
  const uint8_t* Wp;
  const float* gamma;
  const int8_t* xq;
  const float* s;
  float* y;
  int32_t* acc;
  int64_t M, N, K;
  int rows_per_cta;
  int relu2;
};

// Byte offset of entry (nib, i, u, v); the nibble stride is 8 KB, the pair
// stride 1 KB, and the (u, v) part stays below 1 KB.
constexpr uint32_t kNibStride = 16u * 4u * kL4;  // 8192
constexpr uint32_t kPairStride = 8u * kL4;       // 1024
__device__ __forceinline__ uint32_t table_offset(uint32_t nib, int i, int u, int v) {
  return nib * kNibStride + (uint32_t)i * kPairStride + (uint32_t)(u >> 1) * (4u * kL4) + 4u * (uint32_t)v +
         2u * (uint32_t)(u & 1);
}

// Activation j (0, 1) of pair i of the 16 activations in 16-byte word x,
// for pairs of the half ih (i = 4 ih + ii).
__device__ __forceinline__ int pair_x(const uint4& x, int ih, int ii, int j) {
  const uint32_t w = ih ? (ii < 2 ? x.z : x.w) : (ii < 2 ? x.x : x.y);
  return (int)(int8_t)((w >> (16 * (ii & 1) + 8 * j)) & 0xffu);
}

__device__ __forceinline__ void load_row(uint4* pw, const uint4* wrow, int lane, int L4) {
#pragma unroll
  for (int j = 0; j < kWordsPerLane; ++j) {
    const int v = lane + 32 * j;
    pw[j] = v < L4 ? __ldg(wrow + v) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(kLutThreads, 1) gemv_lut_kernel(const LutCfg c) {
  extern __shared__ __align__(16) uint8_t smem[];
  int32_t* acc_sm = reinterpret_cast<int32_t*>(smem + kTableBytes);  // [rows_per_cta]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = (int64_t)blockIdx.x * c.rows_per_cta;
  const int nrows = (int)min((int64_t)c.rows_per_cta, c.N - row0);
  if (nrows <= 0) return;
  const int64_t row_bytes = c.K / 4;
  const float gamma = __ldg(c.gamma);

  for (int64_t m = 0; m < c.M; ++m) {
    for (int r = threadIdx.x; r < nrows; r += kLutThreads) acc_sm[r] = 0;
    const int8_t* x = c.xq + m * c.K;
    for (int64_t k0 = 0; k0 < c.K; k0 += kSliceK) {
      const int ks = (int)min((int64_t)kSliceK, c.K - k0);  // a multiple of 64
      const int L4 = ks / 64;                                // words of the slice in a row
      __syncthreads();  // the previous slice's lookups are done with the tables
      // Tables: thread t takes words 4 v + 2 h and 4 v + 2 h + 1 (v = t % 128,
      // h = (t / 128) % 2) and the pairs i of half t / 256, and stores the two
      // words' entries of a (nib, i) as one 32-bit word.
      {
        const int t = threadIdx.x, v = t & 127, h = (t >> 7) & 1, ih = t >> 8;
        if (v < L4) {
          const uint4* xs = reinterpret_cast<const uint4*>(x + k0) + 4 * v + 2 * h;
          const uint4 a = __ldg(xs), b = __ldg(xs + 1);
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) {
            const int i = 4 * ih + ii;
            const int a0 = pair_x(a, ih, ii, 0), a1 = pair_x(a, ih, ii, 1);
            const int b0 = pair_x(b, ih, ii, 0), b1 = pair_x(b, ih, ii, 1);
#pragma unroll
            for (int nib = 0; nib < 16; ++nib) {
              const int c0 = (nib & 3) - 1, c1 = (nib >> 2) - 1;
              const uint32_t lo = (uint32_t)(c0 * a0 + c1 * a1) & 0xffffu;
              const uint32_t hi = (uint32_t)(c0 * b0 + c1 * b1) << 16;
              *reinterpret_cast<uint32_t*>(smem + table_offset((uint32_t)nib, i, 2 * h, v)) = lo | hi;
            }
          }
        }
      }
      __syncthreads();
      // Lookups: warp-per-row, the next row's words loaded ahead.
      const uint4* wbase = reinterpret_cast<const uint4*>(c.Wp + row0 * row_bytes + k0 / 4);
      const int64_t row_words = row_bytes / 16;
      uint4 cur[kWordsPerLane], nxt[kWordsPerLane];
      if (warp < nrows) load_row(cur, wbase + warp * row_words, lane, L4);
      for (int r = warp; r < nrows; r += kLutWarps) {
        if (r + kLutWarps < nrows) load_row(nxt, wbase + (r + kLutWarps) * row_words, lane, L4);
        int32_t sum = 0;
#pragma unroll
        for (int j = 0; j < kWordsPerLane; ++j) {
          const int v = lane + 32 * j;
          if (v < L4) {
            const uint32_t pk[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t base = table_offset(0u, 0, u, v);  // < 1 KB
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                // nibble i of pk[u] moved to bit 13 (the nibble stride), or-ed with the (u, v) base;
                // the pair's offset i KB stays below the nibble stride
                const uint32_t sh = 4 * i <= 13 ? pk[u] << (13 - 4 * i) : pk[u] >> (4 * i - 13);
                const uint32_t off = (sh & (15u << 13)) | base;
                sum += *reinterpret_cast<const int16_t*>(smem + off + (uint32_t)i * kPairStride);
              }
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) acc_sm[r] += sum;
#pragma unroll
        for (int j = 0; j < kWordsPerLane; ++j) cur[j] = nxt[j];
      }
    }
    __syncthreads();
    const float t = __fdiv_rn(gamma, __ldg(c.s + m));
    for (int r = threadIdx.x; r < nrows; r += kLutThreads) {
      const int64_t o = m * c.N + row0 + r;
      c.y[o] = out_act(__fmul_rn(__int2float_rn(acc_sm[r]), t), c.relu2);
      if (c.acc) c.acc[o] = acc_sm[r];
    }
  }
}

}  // namespace

cudaError_t launch_gemv_lut(const ForwardArgs& a, int num_sms, cudaStream_t stream) {
  const int grid = (int)(a.N < num_sms ? a.N : num_sms);
  LutCfg c{a.Wp, a.gamma, a.xq, a.s, a.y, a.acc, a.M, a.N, a.K, 0, a.relu2 ? 1 : 0};
  c.rows_per_cta = (int)((a.N + grid - 1) / grid);
  const size_t smem = kTableBytes + (size_t)c.rows_per_cta * sizeof(int32_t);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gemv_lut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gemv_lut_kernel<<<grid, kLutThreads, smem, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace bl
