// internal.h -- host-side declarations shared between the C-ABI layer and the
// kernel translation units of libbitlinear.so.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cstdint>
#include <cuda_runtime.h>

#include "bitlinear.h"

namespace bl {

// Per-context facts (context_cache.cu).  `lookup` returns the device address
// of one of the library's __device__ arrays in the current context (it must
// call cudaGetSymbolAddress in the translation unit that defines the array);
// its result is cached per context id and slot, with the current device's SM
// count.  Slots: kSlotErrorWord, kSlotPackScratch.
using SymbolLookup = cudaError_t (*)(void**);
constexpr int kSlotErrorWord = 0;
constexpr int kSlotPackScratch = 1;
constexpr int kCtxSlots = 2;
bl_status context_facts(int slot, SymbolLookup lookup, int* num_sms, void** addr);

// TMA tensor maps (tensor_map.cu).  u8 [outer, inner] row-major, box
// {box_inner bytes, box_outer rows}, swizzle 0 (none), 32, 64 or 128 bytes;
// fp16 [outer, inner] row-major, box {64 elements, box_outer}, 128-byte swizzle.
bool encode_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                  uint32_t box_outer, int swizzle_bytes);
bool encode_f16_2d_sw128(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer);

// Device workspace of bitlinear_pack_weights.
struct PackWorkspace {
  unsigned long long bucket[32];  // exact per-exponent-group sums of |w| (see pack.cu)
  uint32_t nonfinite;             // set if any weight is inf or NaN
  uint32_t thresh_bits;           // fp32 bits of the zero-band threshold T
  float gamma;                    // copy of gamma for later kernels
  uint32_t pad;
};
static_assert(sizeof(PackWorkspace) == 272, "workspace layout");
constexpr size_t kPackWorkspaceBytes = 512;

cudaError_t launch_pack(const float* W, uint64_t n, float eps, uint8_t* Wp, float* gamma, PackWorkspace* ws,
                        int num_sms, cudaStream_t stream);

// The same gamma and ternarisation, written in the base-3 format (five
// weights per byte, rows of `pitch` bytes).  K % 4 == 0.
cudaError_t launch_pack_tq5(const float* W, int64_t N, int64_t K, int64_t pitch, float eps, uint8_t* Wt,
                            float* gamma, PackWorkspace* ws, int num_sms, cudaStream_t stream);

// Per-token quantisation.  From 256 tokens up (K % 16 == 0, 16-byte aligned
// buffers) a persistent kernel with rows staged in shared memory by bulk
// copies, one team of warps per row; else one CTA per row.  err: the device
// error word (the staged kernel's waits are bounded).
cudaError_t launch_quant_act(const void* X, bool bf16, int64_t M, int64_t K, int8_t* xq, float* s, int num_sms,
                             uint32_t* err, cudaStream_t stream, bool test_stall = false);

// Sub-layer RMS normalisation, then the quantisation: r = fp32 sqrt(fp32(ms + eps))
// with ms the exact mean of X^2 rounded once, x_n = fp32(fp32(X * gain) / r), and
// x_q, s the per-token quantisation of x_n.  gain may be null (all ones).
cudaError_t launch_rmsnorm_quant_act(const void* X, bool bf16, int64_t M, int64_t K, const float* gain, float eps,
                                     int8_t* xq, float* s, cudaStream_t stream);

// The RMS-norm quantisation, also writing a tensor-core GEMM's activation
// operand: the fp16 image (x16 at the start of the stream-K workspace, cnt as
// in launch_quant_act_x16) or the fp8 split (in the fp8 GEMM's workspace, as
// launch_quant_act_x8).  X, gain and xq 16-byte aligned, K % 16 == 0.
cudaError_t launch_rmsnorm_quant_act_x16(const void* X, bool bf16, int64_t M, int64_t K, const float* gain, float eps,
                                         int8_t* xq, float* s, void* x16, uint32_t* cnt, int ncnt,
                                         cudaStream_t stream);
cudaError_t launch_rmsnorm_quant_act_x8(const void* X, bool bf16, int64_t M, int64_t K, const float* gain, float eps,
                                        int8_t* xq, float* s, void* ws, int num_sms, cudaStream_t stream);

// The per-token quantisation, also writing the GEMM's fp16 activation operand
// (M x K halves at x16, 16-byte aligned; K % 16 == 0); the first CTA zeroes
// cnt[0 .. ncnt), the stream-K GEMM's arrival counters (cnt may be null).
cudaError_t launch_quant_act_x16(const void* X, bool bf16, int64_t M, int64_t K, int8_t* xq, float* s, void* x16,
                                 uint32_t* cnt, int ncnt, cudaStream_t stream);

struct ForwardArgs {
  const uint8_t* Wp;
  const float* gamma;
  const int8_t* xq;
  const float* s;
  int64_t M, N, K;
  float* y;
  int32_t* acc;
  uint32_t* err;  // device error word
  bool relu2 = false;  // epilogue applies the squared ReLU
  bool test_stall = false;  // test hook: the kernel's copy producer issues nothing, so its bounded waits expire
};

// The forward from base-3 packed weights (five per byte, rows of `pitch`
// bytes), for any M in passes of up to 4 tokens; K % 16 == 0, K <= 40960.
cudaError_t launch_gemv_tq5(const ForwardArgs& a, int64_t pitch, int num_sms, cudaStream_t stream);

// The GEMV by table lookup (gemv_lut.cu): 16-entry tables per pair of
// activations, indexed by the nibbles of the packed weights; any M (the
// weights are read once per token), K % 64 == 0.
cudaError_t launch_gemv_lut(const ForwardArgs& a, int num_sms, cudaStream_t stream);

// Streaming GEMV for a few tokens (tokens are taken in groups of <= 4; K <= 32768).
// pdl: launched as a programmatic dependent of the preceding kernel (the weight
// stream starts before that kernel ends; activations are read after it).
cudaError_t launch_gemv(const ForwardArgs& a, int num_sms, cudaStream_t stream, bool pdl = false);

// Rows of at most this many activations are quantised inside the fused GEMV
// (every CTA reads the row for the maximum); longer rows are quantised by the
// per-token kernel first, and the GEMV follows as its programmatic dependent.
constexpr int64_t kGemvFusedMaxK = 16384;

// The same GEMV with the per-token activation quantisation fused in: reads X
// (bf16 or fp32) instead of x_q / s; the first CTA writes x_q and s out.
// With pdl, launched as a programmatic dependent of the preceding kernel.
cudaError_t launch_gemv_fused(const ForwardArgs& a, const void* X, bool x_bf16, int8_t* xq_out, float* s_out,
                              bool pdl, bool test_stall, int num_sms, cudaStream_t stream);

constexpr int64_t kGemvMaxTokens = 4;
constexpr int64_t kGemvMaxK = 32768;
constexpr int64_t kTq5MaxK = 40960;  // 16 K slices x 32 lanes x 4 words x 20 weights

// fp8 tensor-core GEMM (gemm_f8.cu) for up to kF8MaxTokens tokens (in tiles
// of at most kF8MaxTile), through a
// workspace of gemm_f8_workspace_bytes(M, K, num_sms) bytes (16-byte aligned)
// that holds the e4m3 activation operand (2 rows per token), partial-sum
// slots, arrival counters and every token's sum of activations.  The
// operand, the sums and the zeroed counters come from
// launch_x8_prepass (from x_q) or launch_quant_act_x8 (from X), in stream
// order before launch_gemm_f8.
constexpr int64_t kF8MaxTokens = 64;  // the kernel handles up to 2 tiles of 96; past 64 tokens the f16 GEMM is faster
constexpr int kF8MaxTile = 96;
bool gemm_f8_serves(int64_t M, int64_t N, int64_t K);
int gemm_f8_token_tile(int64_t M);   // tokens per tile: M split into tiles of <= 96, rounded up to 16
int64_t gemm_f8_kblocks(int64_t K);  // 512-k blocks of the operand: ceil(K / 512)
size_t gemm_f8_workspace_bytes(int64_t M, int64_t K, int num_sms);
cudaError_t launch_x8_prepass(const int8_t* xq, int64_t M, int64_t K, void* ws, int num_sms, cudaStream_t stream);
cudaError_t launch_gemm_f8(const ForwardArgs& a, void* ws, int num_sms, cudaStream_t stream);
uint32_t* f8_counters(void* ws, int64_t M, int64_t K, int num_sms);
int32_t* f8_sums(void* ws, int64_t M, int64_t K, int num_sms);  // per token (padded): the sum of its activations
uint8_t* f8_operand(void* ws);
// The per-token quantisation, also writing the fp8 operand (and zeroing the
// counters) of the workspace; K % 16 == 0.
cudaError_t launch_quant_act_x8(const void* X, bool bf16, int64_t M, int64_t K, int8_t* xq, float* s, void* ws,
                                int num_sms, cudaStream_t stream);

// Stream-K fp16 tensor-core GEMM (gemm_f16_sk.cu) for more than
// kF8MaxTokens tokens, in token tiles of at most kSkMaxTile, through a
// workspace of gemm_sk_workspace_bytes(M, K, num_sms) bytes (16-byte aligned):
// the fp16 activation operand (M x K halves at its start), partial-sum slots
// and arrival counters.  The operand and the zeroed counters come from
// launch_x16_sk_prepass (from x_q) or launch_quant_act_x16 with
// sk_counters(...) and num_sms counters (from X), in stream order before
// launch_gemm_f16_sk.
constexpr int kSkMaxTile = 192;
int gemm_sk_token_tile(int64_t M);  // tokens per tile: M split into tiles of <= 192, rounded up to 16
size_t gemm_sk_workspace_bytes(int64_t M, int64_t K, int num_sms);
uint32_t* sk_counters(void* ws, int64_t M, int64_t K, int num_sms);
cudaError_t launch_x16_sk_prepass(const int8_t* xq, int64_t M, int64_t K, void* ws, int num_sms, cudaStream_t stream);
cudaError_t launch_gemm_f16_sk(const ForwardArgs& a, void* ws, int num_sms, cudaStream_t stream);

// Tensor-core GEMM (tcgen05) for more tokens than the GEMV handles well.
cudaError_t launch_gemm_tc(const ForwardArgs& a, int num_sms, cudaStream_t stream);

// The same GEMM on activations expanded to fp16 once per call (M x K halves
// at x16, written by the quantisation kernel or the stream-K GEMM's prepass):
// the persistent one-CTA-per-SM kernel.  It serves the shapes where whole
// output tiles (token tiles of up to 256) fill the SMs at least twice over,
// gemm_x16_persistent_serves; the stream-K GEMM serves the rest.
bool gemm_x16_persistent_serves(int64_t M, int64_t N, int num_sms);
cudaError_t launch_gemm_tc_x16(const ForwardArgs& a, const void* x16, int num_sms, cudaStream_t stream);

}  // namespace bl
