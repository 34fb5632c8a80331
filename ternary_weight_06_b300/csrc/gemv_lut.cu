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
// tables of the current token and slice, then its warps stream their rows:
// lane l of a warp loads 16-byte words l, l + 32, ... of the row's slice and
// looks up its 32 nibbles.  The table index is laid out so that, for any
// codes, the 32 lanes of a lookup touch 32 consecutive 16-bit entries:
//     entry (nib, i, u, v) at ((nib * 8 + i) * 4 + u) * L4 + v,
// for pair p = 8 w + i of 32-bit word w = 4 v + u of the slice (L4 16-byte
// words in the slice), so a lookup is free of bank conflicts.  Row sums are
// reduced across the warp and kept per CTA; the epilogue is that of every
// forward kernel: y = fp32(fp32(acc) * fp32(gamma / s[m])).
// The weights are read once per token.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace bl {
namespace {

constexpr int kLutThreads = 256;
constexpr int kLutWarps = kLutThreads / 32;
constexpr int kSliceK = 8192;                         // activations per table slice
constexpr int kTableBytes = 16 * (kSliceK / 2) * 2;   // 128 KB of int16 entries

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

__device__ __forceinline__ int table_index(int nib, int i, int u, int v, int L4) {
  return ((nib * 8 + i) * 4 + u) * L4 + v;
}

__global__ void __launch_bounds__(kLutThreads, 1) gemv_lut_kernel(const LutCfg c) {
  extern __shared__ __align__(16) uint8_t smem[];
  int16_t* T = reinterpret_cast<int16_t*>(smem);
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
      const int L4 = ks / 64;                                // 16-byte words of packed weights in the slice
      __syncthreads();  // the previous slice's lookups are done with the tables
      // tables: thread t takes the 16 activations of 32-bit word w = t of the slice (8 pairs)
      for (int w = threadIdx.x; w < ks / 16; w += kLutThreads) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + k0) + w);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const int u = w & 3, v = w >> 2;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int x0 = (int)(int8_t)((xw[i >> 1] >> (16 * (i & 1))) & 0xffu);
          const int x1 = (int)(int8_t)((xw[i >> 1] >> (16 * (i & 1) + 8)) & 0xffu);
#pragma unroll
          for (int nib = 0; nib < 16; ++nib)
            T[table_index(nib, i, u, v, L4)] = (int16_t)(((nib & 3) - 1) * x0 + ((nib >> 2) - 1) * x1);
        }
      }
      __syncthreads();
      // lookups: warp-per-row, lane l takes 16-byte words l, l + 32, ... of the row's slice
      for (int r = warp; r < nrows; r += kLutWarps) {
        const uint4* wrow = reinterpret_cast<const uint4*>(c.Wp + (row0 + r) * row_bytes + k0 / 4);
        int32_t sum = 0;
        for (int v = lane; v < L4; v += 32) {
          const uint4 pw = __ldg(wrow + v);
          const uint32_t pk[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) sum += T[table_index((int)((pk[u] >> (4 * i)) & 15u), i, u, v, L4)];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) acc_sm[r] += sum;
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
