// context_cache.cu -- per-context facts the entry points need on the host:
// the SM count of the current device and the device addresses of the
// library's __device__ arrays (the error word, the packing scratch).
//
// A __device__ array has a different address in every CUDA context, and a
// context that was destroyed (cudaDeviceReset) takes its addresses with it.
// So the cache is keyed on the context's unique id (cuCtxGetId: never reused
// within a process), not on the device number: a reset device, or another
// context made current by a host that manages its own contexts, misses the
// cache and gets a fresh lookup, made with that context current.  A hit costs
// two driver queries and a table scan under a mutex; no call here allocates.
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace bl {
namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static std::once_flag once;
  static DriverFns fns;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return fns;
}

struct Entry {
  unsigned long long id = 0;  // 0: unused
  uint64_t last_use = 0;
  int num_sms = 0;
  void* addr[kCtxSlots] = {};
};

constexpr int kEntries = 64;
std::mutex g_mu;
Entry g_entries[kEntries];
uint64_t g_clock = 0;

// Id of the current context; a runtime call that needs a context is made
// first if none is current (the runtime then binds the device's primary one).
bl_status current_context_id(SymbolLookup init, unsigned long long* id) {
  const DriverFns& f = driver_fns();
  if (!f.get_current || !f.get_id) return BL_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return BL_ERR_CUDA;
  if (!ctx) {
    void* p = nullptr;
    if (init(&p) != cudaSuccess) return BL_ERR_CUDA;
    if (f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return BL_ERR_CUDA;
  }
  return f.get_id(ctx, id) == CUDA_SUCCESS && *id != 0 ? BL_OK : BL_ERR_CUDA;
}

}  // namespace

bl_status context_facts(int slot, SymbolLookup lookup, int* num_sms, void** addr) {
  if (slot < 0 || slot >= kCtxSlots || !lookup) return BL_ERR_INVALID_ARG;
  unsigned long long id = 0;
  if (bl_status st = current_context_id(lookup, &id)) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  Entry* e = nullptr;
  for (Entry& c : g_entries)
    if (c.id == id) {
      e = &c;
      break;
    }
  if (!e) {
    // a new context: take a free entry, else the least recently used one
    e = &g_entries[0];
    for (Entry& c : g_entries) {
      if (c.id == 0) {
        e = &c;
        break;
      }
      if (c.last_use < e->last_use) e = &c;
    }
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      return BL_ERR_CUDA;
    *e = Entry{};
    e->id = id;
    e->num_sms = sms;
  }
  if (!e->addr[slot]) {
    void* p = nullptr;
    if (lookup(&p) != cudaSuccess || !p) return BL_ERR_CUDA;
    e->addr[slot] = p;
  }
  e->last_use = ++g_clock;
  if (num_sms) *num_sms = e->num_sms;
  if (addr) *addr = e->addr[slot];
  return BL_OK;
}

}  // namespace bl
