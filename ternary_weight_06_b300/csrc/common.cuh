// common.cuh -- small inline-PTX helpers shared by the BitLinear kernels
// (sm_103a): bounded mbarrier waits, bulk async copies, proxy fences.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace bl {

// Bits of the device error word (see bitlinear_check_device_error).
enum : uint32_t {
  kErrGemvFullWait = 1u << 0,
  kErrGemvEmptyWait = 1u << 1,
  kErrGemmWait = 1u << 2,
  kErrQuantWait = 1u << 3,
};

// A bounded wait gives up after this many nanoseconds of polling.  Every
// legitimate wait in these kernels lasts microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return done != 0;
}

// As mbar_try_wait, but the thread may be suspended in hardware for up to
// `hint_ns` while the phase is incomplete instead of returning at once, so a
// polling loop built on it does not take issue slots from working warps.
// It returns as soon as the phase completes.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar_addr, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Suspend-time hint of the polling loops below.
constexpr uint32_t kWaitHintNs = 20000;

// Waits for the phase with the given parity to complete.  Returns false (and
// records `code` in the error word) if it does not complete within
// kWaitLimitNs; the caller then abandons its work without touching the
// stage.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(a, parity, kWaitHintNs)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, code);
      return false;
    }
  }
}

// 1-D bulk copy global -> shared, completion counted on `bar` (tx bytes).
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: wait until the preceding grid's memory is
// visible (no-op when the kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// Sets a kernel's dynamic shared memory limit and asks for the largest
// shared-memory carveout, so that as many CTAs as the shared memory allows
// are resident per SM (the default carveout can leave room for only one).
template <typename Kernel>
inline cudaError_t set_smem_attrs(Kernel kern, size_t smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

// Output activation of the epilogue: y, or the squared ReLU fp32(max(y,0)^2).
__device__ __forceinline__ float out_act(float y, int relu2) {
  if (relu2) {
    const float r = y > 0.0f ? y : 0.0f;
    return __fmul_rn(r, r);
  }
  return y;
}

// ---- exact int8 -> fp16 operand expansion (shared by the GEMM and the
// activation quantisation, which can write the GEMM's operand directly)

// Two fp16 of 1024 + byte, from bytes b0, b1 of w (selector 0x4140) or b2, b3 (0x4342).
__device__ __forceinline__ uint32_t bytes_to_h2(uint32_t w, uint32_t sel) { return __byte_perm(w, 0x64646464u, sel); }

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 16 ternary codes (one packed word, k = 0..15 at bits 2k) -> 16 fp16 of
// code - 1 as 8 pairs, positions p = 4 i + j holding k = 4 j + i: byte j of
// (P >> 2i) & 0x03030303 is the code of k = 4 j + i.
__device__ __forceinline__ void unpack16_f16(uint32_t P, uint32_t* h /* 8 words */) {
  const uint32_t k1025 = 0x64016401u;  // fp16 (1025, 1025): 1024 + code - 1025 = code - 1
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t S = (P >> (2 * i)) & 0x03030303u;
    h[2 * i] = h2_sub(bytes_to_h2(S, 0x4140), k1025);
    h[2 * i + 1] = h2_sub(bytes_to_h2(S, 0x4342), k1025);
  }
}

// 16 int8 activations (natural order, 4 words) -> 16 fp16 in order p = 4i + j.
__device__ __forceinline__ void convert_x16_f16(uint4 v, uint32_t* h /* 8 words */) {
  const uint32_t x0 = v.x ^ 0x80808080u, x1 = v.y ^ 0x80808080u, x2 = v.z ^ 0x80808080u, x3 = v.w ^ 0x80808080u;
  const uint32_t t0 = __byte_perm(x0, x1, 0x5140), t1 = __byte_perm(x2, x3, 0x5140);
  const uint32_t t2 = __byte_perm(x0, x1, 0x7362), t3 = __byte_perm(x2, x3, 0x7362);
  const uint32_t o[4] = {__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632), __byte_perm(t2, t3, 0x5410),
                         __byte_perm(t2, t3, 0x7632)};
  const uint32_t k1152 = 0x64806480u;  // fp16 (1152, 1152): undoes the +128 bias and the 1024 offset
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[2 * i] = h2_sub(bytes_to_h2(o[i], 0x4140), k1152);
    h[2 * i + 1] = h2_sub(bytes_to_h2(o[i], 0x4342), k1152);
  }
}

// ---- e4m3 activation operand of the fp8 GEMM (shared by the GEMM's prepass
// and the activation quantisation, which can write the operand directly)

// e4m3 bits of v * 2^-d for an integer v with 1 <= |v| <= 15 (or 0) and
// d in {0, 2}: exponent from the top bit, the three bits below it as the
// mantissa; every such value is a normal e4m3 number, exactly.
__device__ __forceinline__ uint32_t e4m3_small(int v, int d) {
  if (v == 0) return 0u;
  const uint32_t s = v < 0 ? 0x80u : 0u;
  const uint32_t a = (uint32_t)(v < 0 ? -v : v);
  const uint32_t e = 31u - __clz(a);
  return s | ((e + 7u - (uint32_t)d) << 3) | (((a << 3) >> e) & 7u);
}

// 16 int8 activations (natural k order, 4 words) -> the token's two e4m3
// operand rows of the fp8 GEMM, h and l (x = 16 h + l, h = x >> 4 in
// [-8, 7], l = x & 15), 16 bytes each.  Position p = 4 i + j of a row holds
// k = 4 j + i: the order in which the GEMM expands a packed weight word by
// masks.  The weight bytes at odd i carry 4 c (the code shifted by two bits),
// so the activation there is h / 4 or l / 4 (exact in e4m3).
__device__ __forceinline__ void x8_rows16(uint4 v, uint4* hi, uint4* lo) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t H[4] = {0u, 0u, 0u, 0u}, L[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int x = (int)(int8_t)((w[k >> 2] >> (8 * (k & 3))) & 0xffu);
    const int i = k & 3, j = k >> 2, d = (i & 1) ? 2 : 0;  // word i, byte j of the row's 16 bytes
    H[i] |= e4m3_small(x >> 4, d) << (8 * j);
    L[i] |= e4m3_small(x & 15, d) << (8 * j);
  }
  *hi = make_uint4(H[0], H[1], H[2], H[3]);
  *lo = make_uint4(L[0], L[1], L[2], L[3]);
}

// Sum of the 16 int8 values of a group (4 words).
__device__ __forceinline__ int sum16_i8(uint4 v) {
  return __dp4a((int)v.w, 0x01010101, __dp4a((int)v.z, 0x01010101, __dp4a((int)v.y, 0x01010101, __dp4a((int)v.x, 0x01010101, 0))));
}

// The sum of v over the CTA, written by thread 0 to *dst.  Every thread of
// the CTA calls it once (blockDim.x a multiple of 32).
__device__ __forceinline__ void block_sum_store(int v, int32_t* dst) {
  __shared__ int part[32];
  v = __reduce_add_sync(0xffffffffu, v);
  if ((threadIdx.x & 31u) == 0u) part[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32u) {
    int w = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0;
    w = __reduce_add_sync(0xffffffffu, w);
    if (threadIdx.x == 0u) *dst = w;
  }
}

// Tiled layout of that operand: blocks of BN tokens x kX8Block k, each block
// NB = 2 BN rows (h and l of every token) of kX8Block bytes stored as four
// 128-byte-wide boxes [NB rows][128 B] one after another, with the 128-byte
// swizzle of the MMA's shared-memory operands applied (16-byte chunk c of row
// j at chunk c ^ (j & 7)); block (token tile mt, k-block kb) starts at byte
// (mt * nkb + kb) * NB * kX8Block.  One contiguous copy of a block gives the
// shared-memory image the MMA reads.  Rows of tokens past M and bytes of k
// past K are zero.
constexpr int kX8Block = 512;

// Every token's sum of activations comes in partial sums over 4096-k chunks
// (the last one short): x8_sum_parts(K) int32 per token, token-major.
constexpr int kX8SumK = 4096;
__host__ __device__ __forceinline__ int x8_sum_parts(int64_t K) { return (int)((K + kX8SumK - 1) / kX8SumK); }

// Byte offset of the 16-byte group of k = k16 .. k16 + 15 (k16 % 16 == 0) in
// row hl (0: h, 1: l) of token m.
__device__ __forceinline__ size_t x8_group_offset(int64_t m, int64_t k16, int hl, int BN, int64_t nkb) {
  const int64_t mt = m / BN, kb = k16 / kX8Block;
  const int t = (int)(m - mt * BN), kk = (int)(k16 - kb * kX8Block);
  const int NB = 2 * BN, j = 2 * t + hl, c = (kk & 127) >> 4;
  return (size_t)(mt * nkb + kb) * (size_t)(NB * kX8Block) + (size_t)((kk >> 7) * NB * 128 + j * 128 + ((c ^ (j & 7)) << 4));
}

}  // namespace bl
