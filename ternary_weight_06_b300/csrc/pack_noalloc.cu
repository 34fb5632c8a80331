// pack_noalloc.cu -- bitlinear_pack_weights_noalloc: weight packing for
// callers that cannot hand the library any device memory of its own.
//
// bitlinear_pack_weights needs a small device workspace (the exact |W| sums
// and the zero-band threshold).  Some callers cannot provide one: a host
// application whose device memory is owned by its own pool allocator (an
// extra cudaMalloc would fail or fragment that pool), and plug-in hosts that
// only pass pointers to memory somebody else owns.  This
// entry point therefore keeps the workspace in a fixed array inside the
// library's device image instead, so it allocates nothing.
//
// The array lives in every GPU that loads the library until the process
// exits.  Host code cannot use its name as a device address: the address is
// looked up with cudaGetSymbolAddress, in this file, with the device's
// context current, and cached per CUDA context (context_cache.cu), because
// each context has its own copy of the array and a reset device's context is
// a new one.
#include <cmath>
#include <cstdint>

#include "bitlinear.h"
#include "internal.h"

namespace {

// Capacity of the shared scratch.  The packing kernels need
// sizeof(bl::PackWorkspace) bytes whatever N and K are.
constexpr size_t kScratchBytes = 512;
static_assert(sizeof(bl::PackWorkspace) <= kScratchBytes, "scratch too small for the pack workspace");

static __device__ __align__(256) unsigned char g_pack_scratch[kScratchBytes];

cudaError_t lookup_scratch(void** p) { return cudaGetSymbolAddress(p, g_pack_scratch); }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" bl_status bitlinear_pack_weights_noalloc(const float* W, int64_t N, int64_t K, float eps,
                                                    uint8_t* W_packed, float* gamma, cudaStream_t stream) {
  if (!W || !W_packed || !gamma) return BL_ERR_INVALID_ARG;
  if (N < 1 || K < 1) return BL_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || !(eps > 0.0f)) return BL_ERR_INVALID_ARG;
  if (K % 4 != 0 || K < 4) return BL_ERR_UNSUPPORTED_SHAPE;
  if (N > (int64_t)(1ull << 32) / K) return BL_ERR_UNSUPPORTED_SHAPE;  // N*K <= 2^32
  if (!aligned(W, 16) || !aligned(W_packed, 16) || !aligned(gamma, 4)) return BL_ERR_MISALIGNED;
  // The scratch cannot grow: refuse any request that would need more than it holds.
  if (bitlinear_pack_workspace_bytes(N, K) > kScratchBytes) return BL_ERR_WORKSPACE;
  int num_sms = 0;
  void* scratch = nullptr;
  if (bl_status st = bl::context_facts(bl::kSlotPackScratch, lookup_scratch, &num_sms, &scratch)) return st;
  // launch_pack clears the workspace on `stream` before its kernels use it.
  const cudaError_t e = bl::launch_pack(W, (uint64_t)N * (uint64_t)K, eps, W_packed, gamma,
                                        static_cast<bl::PackWorkspace*>(scratch), num_sms, stream);
  return e == cudaSuccess ? BL_OK : BL_ERR_CUDA;
}
