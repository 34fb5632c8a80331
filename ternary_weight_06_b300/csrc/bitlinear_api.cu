// bitlinear_api.cu -- the extern "C" entry points of libbitlinear.so: argument
// validation on the host, kernel selection, and the device error word.
// Contracts are documented in include/bitlinear.h.
#include <cmath>
#include <cstdint>

#include "bitlinear.h"
#include "internal.h"

// The library's only state: one error word per device, set by kernels whose
// bounded waits expire (see bitlinear_check_device_error).
static __device__ uint32_t g_bl_error_word;

namespace {

struct DeviceInfo {
  int num_sms = 0;
  uint32_t* err = nullptr;
};

cudaError_t lookup_error_word(void** p) { return cudaGetSymbolAddress(p, g_bl_error_word); }

// Facts of the current context: SM count and the error word's address.
bl_status device_info(DeviceInfo* out) {
  void* p = nullptr;
  if (bl_status st = bl::context_facts(bl::kSlotErrorWord, lookup_error_word, &out->num_sms, &p)) return st;
  out->err = static_cast<uint32_t*>(p);
  return BL_OK;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bl_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BL_OK : BL_ERR_CUDA; }

// The few-token route (M <= 4, K <= 32768): one fused quantise + GEMV kernel
// for rows up to 16384 activations (and always under the stall test hook);
// longer rows are quantised by the per-token kernel, and the GEMV follows as
// its programmatic dependent, its weight stream starting meanwhile.
cudaError_t launch_few_tokens(const bl::ForwardArgs& a, const void* X, bool bf16, int8_t* x_q, float* s,
                              bool resident, bool stall, const DeviceInfo& d, cudaStream_t stream) {
  if (a.K <= bl::kGemvFusedMaxK || stall)
    return bl::launch_gemv_fused(a, X, bf16, x_q, s, resident, stall, d.num_sms, stream);
  if (cudaError_t e = bl::launch_quant_act(X, bf16, a.M, a.K, x_q, s, d.num_sms, d.err, stream)) return e;
  return bl::launch_gemv(a, d.num_sms, stream, true);
}

}  // namespace

extern "C" {

size_t bitlinear_pack_workspace_bytes(int64_t N, int64_t K) {
  (void)N;
  (void)K;
  return bl::kPackWorkspaceBytes;
}

bl_status bitlinear_pack_weights(const float* W, int64_t N, int64_t K, float eps, uint8_t* W_packed, float* gamma,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!W || !W_packed || !gamma || !workspace) return BL_ERR_INVALID_ARG;
  if (N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || !(eps > 0.0f)) return BL_ERR_INVALID_ARG;
  if (K % 4 != 0 || K < 4) return BL_ERR_UNSUPPORTED_SHAPE;
  if (N > (int64_t)(1ull << 32) / K) return BL_ERR_UNSUPPORTED_SHAPE;  // N*K <= 2^32
  if (!aligned(W, 16) || !aligned(W_packed, 16) || !aligned(gamma, 4) || !aligned(workspace, 16))
    return BL_ERR_MISALIGNED;
  if (workspace_bytes < bl::kPackWorkspaceBytes) return BL_ERR_WORKSPACE;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  return from_cuda(bl::launch_pack(W, (uint64_t)N * (uint64_t)K, eps, W_packed, gamma,
                                   static_cast<bl::PackWorkspace*>(workspace), d.num_sms, stream));
}

int64_t bitlinear_tq5_row_bytes(int64_t K) {
  if (K < 1) return 0;
  return ((K + 4) / 5 + 15) / 16 * 16;
}

bl_status bitlinear_pack_weights_tq5(const float* W, int64_t N, int64_t K, float eps, uint8_t* W_tq5, float* gamma,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!W || !W_tq5 || !gamma || !workspace) return BL_ERR_INVALID_ARG;
  if (N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || !(eps > 0.0f)) return BL_ERR_INVALID_ARG;
  if (K % 4 != 0 || K < 4) return BL_ERR_UNSUPPORTED_SHAPE;
  if (N > (int64_t)(1ull << 32) / K) return BL_ERR_UNSUPPORTED_SHAPE;  // N*K <= 2^32
  if (!aligned(W, 16) || !aligned(W_tq5, 16) || !aligned(gamma, 4) || !aligned(workspace, 16))
    return BL_ERR_MISALIGNED;
  if (workspace_bytes < bl::kPackWorkspaceBytes) return BL_ERR_WORKSPACE;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  return from_cuda(bl::launch_pack_tq5(W, N, K, bitlinear_tq5_row_bytes(K), eps, W_tq5, gamma,
                                       static_cast<bl::PackWorkspace*>(workspace), d.num_sms, stream));
}

bl_status bitlinear_forward_tq5(const uint8_t* W_tq5, const float* gamma, const int8_t* x_q, const float* s,
                                int64_t M, int64_t N, int64_t K, float* y, int32_t* acc, unsigned flags,
                                cudaStream_t stream) {
  if (!W_tq5 || !gamma || !x_q || !s || !y) return BL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (flags & ~(BITLINEAR_RELU2 | BITLINEAR_TEST_STALL)) return BL_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > bl::kTq5MaxK || M > INT32_MAX) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_tq5, 16) || !aligned(x_q, 16) || !aligned(y, 16) || !aligned(gamma, 4) || !aligned(s, 4) ||
      (acc && !aligned(acc, 16)))
    return BL_ERR_MISALIGNED;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  if (N > (int64_t)2048 * d.num_sms) return BL_ERR_UNSUPPORTED_SHAPE;  // per-CTA row sums must fit shared memory
  bl::ForwardArgs a{W_tq5, gamma, x_q, s, M, N, K, y, acc, d.err, (flags & BITLINEAR_RELU2) != 0,
                    (flags & BITLINEAR_TEST_STALL) != 0};
  return from_cuda(bl::launch_gemv_tq5(a, bitlinear_tq5_row_bytes(K), d.num_sms, stream));
}

bl_status bitlinear_quant_act(const void* X, bl_dtype dtype, int64_t M, int64_t K, int8_t* x_q, float* s,
                              cudaStream_t stream) {
  if (!X || !x_q || !s) return BL_ERR_INVALID_ARG;
  if (M < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_INVALID_ARG;
  if (M > INT32_MAX || K > (int64_t)1 << 24) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(X, 16) || !aligned(x_q, 16) || !aligned(s, 4)) return BL_ERR_MISALIGNED;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  return from_cuda(bl::launch_quant_act(X, dtype == BL_BF16, M, K, x_q, s, d.num_sms, d.err, stream));
}

bl_status bitlinear_rmsnorm_quant_act(const void* X, bl_dtype dtype, int64_t M, int64_t K, const float* gain,
                                      float eps, int8_t* x_q, float* s, cudaStream_t stream) {
  if (!X || !x_q || !s) return BL_ERR_INVALID_ARG;
  if (M < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || !(eps > 0.0f)) return BL_ERR_INVALID_ARG;
  if (M > INT32_MAX || K > (int64_t)1 << 24) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(X, dtype == BL_BF16 ? 2 : 4) || !aligned(s, 4) || (gain && !aligned(gain, 4))) return BL_ERR_MISALIGNED;
  return from_cuda(bl::launch_rmsnorm_quant_act(X, dtype == BL_BF16, M, K, gain, eps, x_q, s, stream));
}

bl_status bitlinear_forward(const uint8_t* W_packed, const float* gamma, const int8_t* x_q, const float* s,
                            int64_t M, int64_t N, int64_t K, float* y, int32_t* acc, cudaStream_t stream) {
  if (!W_packed || !gamma || !x_q || !s || !y) return BL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (K % 64 != 0 || K > BITLINEAR_MAX_K || M > INT32_MAX || N > INT32_MAX) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_packed, 16) || !aligned(x_q, 16) || !aligned(y, 16) || !aligned(gamma, 4) || !aligned(s, 4) ||
      (acc && !aligned(acc, 16)))
    return BL_ERR_MISALIGNED;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  bl::ForwardArgs a{W_packed, gamma, x_q, s, M, N, K, y, acc, d.err};
  if (M > bl::kGemvMaxTokens || K > bl::kGemvMaxK) return from_cuda(bl::launch_gemm_tc(a, d.num_sms, stream));
  return from_cuda(bl::launch_gemv(a, d.num_sms, stream));
}

bl_status bitlinear_forward_lut(const uint8_t* W_packed, const float* gamma, const int8_t* x_q, const float* s,
                                int64_t M, int64_t N, int64_t K, float* y, int32_t* acc, unsigned flags,
                                cudaStream_t stream) {
  if (!W_packed || !gamma || !x_q || !s || !y) return BL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (flags & ~BITLINEAR_RELU2) return BL_ERR_INVALID_ARG;
  if (K % 64 != 0 || K > BITLINEAR_MAX_K || M > INT32_MAX || N > INT32_MAX) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_packed, 16) || !aligned(x_q, 16) || !aligned(y, 4) || !aligned(gamma, 4) || !aligned(s, 4) ||
      (acc && !aligned(acc, 4)))
    return BL_ERR_MISALIGNED;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  if (N > (int64_t)16384 * d.num_sms) return BL_ERR_UNSUPPORTED_SHAPE;  // per-CTA row sums must fit shared memory
  bl::ForwardArgs a{W_packed, gamma, x_q, s, M, N, K, y, acc, d.err, (flags & BITLINEAR_RELU2) != 0};
  return from_cuda(bl::launch_gemv_lut(a, d.num_sms, stream));
}

bl_status bitlinear_quant_forward(const uint8_t* W_packed, const float* gamma, const void* X, bl_dtype dtype,
                                  int64_t M, int64_t N, int64_t K, float* y, int8_t* x_q, float* s, int32_t* acc,
                                  unsigned flags, cudaStream_t stream) {
  if (!W_packed || !gamma || !X || !y || !x_q || !s) return BL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_INVALID_ARG;
  if (flags & ~(BITLINEAR_WEIGHTS_RESIDENT | BITLINEAR_RELU2 | BITLINEAR_TEST_STALL)) return BL_ERR_INVALID_ARG;
  if (K % 64 != 0 || K > BITLINEAR_MAX_K || M > INT32_MAX || N > INT32_MAX) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_packed, 16) || !aligned(X, 16) || !aligned(x_q, 16) || !aligned(y, 16) || !aligned(gamma, 4) ||
      !aligned(s, 4) || (acc && !aligned(acc, 16)))
    return BL_ERR_MISALIGNED;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  bl::ForwardArgs a{W_packed, gamma, x_q, s, M, N, K, y, acc, d.err, (flags & BITLINEAR_RELU2) != 0};
  const bool stall = (flags & BITLINEAR_TEST_STALL) != 0;
  if (M <= bl::kGemvMaxTokens && K <= bl::kGemvMaxK)
    return from_cuda(launch_few_tokens(a, X, dtype == BL_BF16, x_q, s, (flags & BITLINEAR_WEIGHTS_RESIDENT) != 0,
                                       stall, d, stream));
  a.test_stall = stall;  // the staged quantisation (from 256 tokens) and the GEMM each give up
  if (cudaError_t e = bl::launch_quant_act(X, dtype == BL_BF16, M, K, x_q, s, d.num_sms, d.err, stream, stall))
    return from_cuda(e);
  return from_cuda(bl::launch_gemm_tc(a, d.num_sms, stream));
}

size_t bitlinear_forward_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || K < 1) return 0;
  if (M <= bl::kGemvMaxTokens && K <= bl::kGemvMaxK) return 0;  // the GEMV needs none
  // both tensor-core GEMMs keep partial-sum slots per CTA (one CTA per SM);
  // without a usable device the bound assumes 256 SMs
  DeviceInfo d;
  const int sms = device_info(&d) == BL_OK ? d.num_sms : 256;
  if (bl::gemm_f8_serves(M, N, K)) return bl::gemm_f8_workspace_bytes(M, K, sms);
  return bl::gemm_sk_workspace_bytes(M, K, sms);
}

namespace {

// Checks the workspace of the *_ws calls against the requirement of the path taken.
bl_status check_workspace(int64_t M, int64_t N, int64_t K, const void* workspace, size_t workspace_bytes) {
  const size_t need = bitlinear_forward_workspace_bytes(M, N, K);
  if (need == 0) return BL_OK;
  if (!workspace || workspace_bytes < need) return BL_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return BL_ERR_MISALIGNED;
  return BL_OK;
}

}  // namespace

bl_status bitlinear_forward_ws(const uint8_t* W_packed, const float* gamma, const int8_t* x_q, const float* s,
                               int64_t M, int64_t N, int64_t K, float* y, int32_t* acc, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  if (!W_packed || !gamma || !x_q || !s || !y) return BL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (K % 64 != 0 || K > BITLINEAR_MAX_K || M > INT32_MAX || N > INT32_MAX) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_packed, 16) || !aligned(x_q, 16) || !aligned(y, 16) || !aligned(gamma, 4) || !aligned(s, 4) ||
      (acc && !aligned(acc, 16)))
    return BL_ERR_MISALIGNED;
  if (bl_status st = check_workspace(M, N, K, workspace, workspace_bytes)) return st;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  bl::ForwardArgs a{W_packed, gamma, x_q, s, M, N, K, y, acc, d.err};
  if (M <= bl::kGemvMaxTokens && K <= bl::kGemvMaxK) return from_cuda(bl::launch_gemv(a, d.num_sms, stream));
  if (bl::gemm_f8_serves(M, N, K)) {
    if (cudaError_t e = bl::launch_x8_prepass(x_q, M, K, workspace, d.num_sms, stream)) return from_cuda(e);
    return from_cuda(bl::launch_gemm_f8(a, workspace, d.num_sms, stream));
  }
  if (cudaError_t e = bl::launch_x16_sk_prepass(x_q, M, K, workspace, d.num_sms, stream)) return from_cuda(e);
  if (bl::gemm_x16_persistent_serves(M, N, d.num_sms))
    return from_cuda(bl::launch_gemm_tc_x16(a, workspace, d.num_sms, stream));
  return from_cuda(bl::launch_gemm_f16_sk(a, workspace, d.num_sms, stream));
}

bl_status bitlinear_quant_forward_ws(const uint8_t* W_packed, const float* gamma, const void* X, bl_dtype dtype,
                                     int64_t M, int64_t N, int64_t K, float* y, int8_t* x_q, float* s, int32_t* acc,
                                     unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!W_packed || !gamma || !X || !y || !x_q || !s) return BL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_INVALID_ARG;
  if (flags & ~(BITLINEAR_WEIGHTS_RESIDENT | BITLINEAR_RELU2 | BITLINEAR_TEST_STALL)) return BL_ERR_INVALID_ARG;
  if (K % 64 != 0 || K > BITLINEAR_MAX_K || M > INT32_MAX || N > INT32_MAX) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_packed, 16) || !aligned(X, 16) || !aligned(x_q, 16) || !aligned(y, 16) || !aligned(gamma, 4) ||
      !aligned(s, 4) || (acc && !aligned(acc, 16)))
    return BL_ERR_MISALIGNED;
  if (bl_status st = check_workspace(M, N, K, workspace, workspace_bytes)) return st;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  bl::ForwardArgs a{W_packed, gamma, x_q, s, M, N, K, y, acc, d.err, (flags & BITLINEAR_RELU2) != 0};
  const bool stall = (flags & BITLINEAR_TEST_STALL) != 0;
  if (M <= bl::kGemvMaxTokens && K <= bl::kGemvMaxK)
    return from_cuda(launch_few_tokens(a, X, dtype == BL_BF16, x_q, s, (flags & BITLINEAR_WEIGHTS_RESIDENT) != 0,
                                       stall, d, stream));
  a.test_stall = stall;  // the GEMM gives up
  if (bl::gemm_f8_serves(M, N, K)) {
    if (cudaError_t e = bl::launch_quant_act_x8(X, dtype == BL_BF16, M, K, x_q, s, workspace, d.num_sms, stream))
      return from_cuda(e);
    return from_cuda(bl::launch_gemm_f8(a, workspace, d.num_sms, stream));
  }
  if (cudaError_t e = bl::launch_quant_act_x16(X, dtype == BL_BF16, M, K, x_q, s, workspace,
                                               bl::sk_counters(workspace, M, K, d.num_sms), d.num_sms, stream))
    return from_cuda(e);
  if (bl::gemm_x16_persistent_serves(M, N, d.num_sms))
    return from_cuda(bl::launch_gemm_tc_x16(a, workspace, d.num_sms, stream));
  return from_cuda(bl::launch_gemm_f16_sk(a, workspace, d.num_sms, stream));
}

bl_status bitlinear_quant_forward_requant_ws(const uint8_t* W_packed, const float* gamma, const void* X, bl_dtype dtype,
                                             int64_t M, int64_t N, int64_t K, float* y, int8_t* x_q, float* s,
                                             int8_t* y_q, float* s_y, unsigned flags, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream) {
  if (!W_packed || !gamma || !X || !y || !x_q || !s || !y_q || !s_y) return BL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_INVALID_ARG;
  if (flags & ~BITLINEAR_RELU2) return BL_ERR_INVALID_ARG;
  if (K % 64 != 0 || K > BITLINEAR_MAX_K || M > INT32_MAX || N > INT32_MAX) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_packed, 16) || !aligned(X, 16) || !aligned(x_q, 16) || !aligned(y, 16) || !aligned(gamma, 4) ||
      !aligned(s, 4) || !aligned(y_q, 16) || !aligned(s_y, 4))
    return BL_ERR_MISALIGNED;
  if (bl_status st = check_workspace(M, N, K, workspace, workspace_bytes)) return st;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  bl::ForwardArgs a{W_packed, gamma, x_q, s, M, N, K, y, nullptr, d.err, (flags & BITLINEAR_RELU2) != 0};
  const bool bf16 = dtype == BL_BF16;
  cudaError_t e;
  if (M <= bl::kGemvMaxTokens && K <= bl::kGemvMaxK) {
    e = launch_few_tokens(a, X, bf16, x_q, s, false, false, d, stream);
  } else if (bl::gemm_f8_serves(M, N, K)) {
    e = bl::launch_quant_act_x8(X, bf16, M, K, x_q, s, workspace, d.num_sms, stream);
    if (e == cudaSuccess) e = bl::launch_gemm_f8(a, workspace, d.num_sms, stream);
  } else {
    e = bl::launch_quant_act_x16(X, bf16, M, K, x_q, s, workspace, bl::sk_counters(workspace, M, K, d.num_sms),
                                 d.num_sms, stream);
    if (e == cudaSuccess)
      e = bl::gemm_x16_persistent_serves(M, N, d.num_sms) ? bl::launch_gemm_tc_x16(a, workspace, d.num_sms, stream)
                                                          : bl::launch_gemm_f16_sk(a, workspace, d.num_sms, stream);
  }
  if (e != cudaSuccess) return from_cuda(e);
  // y is still resident in L2 (at most M x N x 4 bytes, written just now): the
  // per-token quantisation reads it back from there
  return from_cuda(bl::launch_quant_act(y, false, M, N, y_q, s_y, d.num_sms, d.err, stream));
}

bl_status bitlinear_rmsnorm_quant_forward_ws(const uint8_t* W_packed, const float* gamma, const void* X, bl_dtype dtype,
                                             int64_t M, int64_t N, int64_t K, const float* gain, float eps, float* y,
                                             int8_t* x_q, float* s, int32_t* acc, unsigned flags, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream) {
  if (!W_packed || !gamma || !X || !y || !x_q || !s) return BL_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || !(eps > 0.0f)) return BL_ERR_INVALID_ARG;
  if (flags & ~BITLINEAR_RELU2) return BL_ERR_INVALID_ARG;
  if (K % 64 != 0 || K > BITLINEAR_MAX_K || M > INT32_MAX || N > INT32_MAX) return BL_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_packed, 16) || !aligned(X, 16) || !aligned(x_q, 16) || !aligned(y, 16) || !aligned(gamma, 4) ||
      !aligned(s, 4) || (gain && !aligned(gain, 16)) || (acc && !aligned(acc, 16)))
    return BL_ERR_MISALIGNED;
  if (bl_status st = check_workspace(M, N, K, workspace, workspace_bytes)) return st;
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  bl::ForwardArgs a{W_packed, gamma, x_q, s, M, N, K, y, acc, d.err, (flags & BITLINEAR_RELU2) != 0};
  const bool bf16 = dtype == BL_BF16;
  if (M <= bl::kGemvMaxTokens && K <= bl::kGemvMaxK) {
    // a few tokens: the RMS-norm quantisation, then the GEMV on x_q
    if (cudaError_t e = bl::launch_rmsnorm_quant_act(X, bf16, M, K, gain, eps, x_q, s, stream)) return from_cuda(e);
    return from_cuda(bl::launch_gemv(a, d.num_sms, stream));
  }
  // more: the RMS-norm quantisation writes the GEMM's operand directly
  if (bl::gemm_f8_serves(M, N, K)) {
    if (cudaError_t e = bl::launch_rmsnorm_quant_act_x8(X, bf16, M, K, gain, eps, x_q, s, workspace, d.num_sms, stream))
      return from_cuda(e);
    return from_cuda(bl::launch_gemm_f8(a, workspace, d.num_sms, stream));
  }
  if (cudaError_t e = bl::launch_rmsnorm_quant_act_x16(X, bf16, M, K, gain, eps, x_q, s, workspace,
                                                       bl::sk_counters(workspace, M, K, d.num_sms), d.num_sms, stream))
    return from_cuda(e);
  if (bl::gemm_x16_persistent_serves(M, N, d.num_sms))
    return from_cuda(bl::launch_gemm_tc_x16(a, workspace, d.num_sms, stream));
  return from_cuda(bl::launch_gemm_f16_sk(a, workspace, d.num_sms, stream));
}

bl_status bitlinear_check_device_error(cudaStream_t stream) {
  DeviceInfo d;
  if (bl_status st = device_info(&d)) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BL_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbolAsync(&word, g_bl_error_word, sizeof(word), 0, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return BL_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BL_ERR_CUDA;
  if (word) {
    if (cudaMemsetAsync(d.err, 0, sizeof(uint32_t), stream) != cudaSuccess) return BL_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BL_ERR_CUDA;
    return BL_ERR_TIMEOUT;
  }
  return BL_OK;
}

const char* bitlinear_status_string(bl_status status) {
  switch (status) {
    case BL_OK: return "BL_OK";
    case BL_ERR_INVALID_ARG: return "BL_ERR_INVALID_ARG: null pointer, non-positive size, bad eps or dtype";
    case BL_ERR_UNSUPPORTED_SHAPE: return "BL_ERR_UNSUPPORTED_SHAPE: a size outside the documented limits";
    case BL_ERR_MISALIGNED: return "BL_ERR_MISALIGNED: a pointer lacks the documented alignment";
    case BL_ERR_WORKSPACE: return "BL_ERR_WORKSPACE: workspace smaller than bitlinear_pack_workspace_bytes()";
    case BL_ERR_CUDA: return "BL_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case BL_ERR_TIMEOUT: return "BL_ERR_TIMEOUT: a kernel gave up on a bounded wait";
  }
  return "unknown bl_status";
}

}  // extern "C"
