// Per-context cache of kernel attributes and cluster occupancy (see launch_cache.h).
//
// A context is identified by the driver's 64-bit context id (cuCtxGetId), which is unique for the
// life of the process, so a context destroyed and re-created at the same handle is not mistaken
// for the old one.  Both driver entry points are looked up once through the runtime.
#include "launch_cache.h"

#include <cuda.h>
#include <stdint.h>

#include <mutex>

namespace specv {
namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver() {
  static DriverFns fns;
  static std::once_flag once;
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

// Id of the calling thread's current context, or 0 when there is none yet (the runtime binds its
// primary context lazily) or the driver cannot say.
unsigned long long current_context_id() {
  const DriverFns& d = driver();
  if (!d.get_current || !d.get_id) return 0;
  CUcontext ctx = nullptr;
  if (d.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (d.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct Entry {
  unsigned long long ctx;
  const void* func;
  long long key;   // attribute entries: 0; occupancy entries: the launch shape
  int value;       // attribute entries: the limit set; occupancy entries: active clusters
};

constexpr int kEntries = 512;
std::mutex g_mu;
Entry g_tab[kEntries];
int g_used = 0, g_next = 0;

Entry* find(unsigned long long ctx, const void* func, long long key) {
  for (int i = 0; i < g_used; ++i)
    if (g_tab[i].ctx == ctx && g_tab[i].func == func && g_tab[i].key == key) return &g_tab[i];
  return nullptr;
}

void put(unsigned long long ctx, const void* func, long long key, int value) {
  Entry* e = find(ctx, func, key);
  if (!e) {
    // a full table overwrites its oldest entry (the cached settings are only ever made again)
    e = &g_tab[g_next];
    g_next = (g_next + 1) % kEntries;
    if (g_used < kEntries) ++g_used;
  }
  *e = Entry{ctx, func, key, value};
}

}  // namespace

cudaError_t ensure_dynamic_smem(const void* func, int bytes) {
  unsigned long long ctx = current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_mu);
    const Entry* e = find(ctx, func, 0);
    if (e && e->value >= bytes) return cudaSuccess;
  }
  const cudaError_t err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err != cudaSuccess) return err;
  if (ctx == 0) ctx = current_context_id();  // the call above has bound the runtime's context
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_mu);
    const Entry* e = find(ctx, func, 0);
    if (!e || e->value < bytes) put(ctx, func, 0, bytes);
  }
  return cudaSuccess;
}

cudaError_t max_active_clusters(int* active, const void* func, const cudaLaunchConfig_t* cfg) {
  unsigned cluster = 1;
  for (unsigned i = 0; i < cfg->numAttrs; ++i)
    if (cfg->attrs[i].id == cudaLaunchAttributeClusterDimension)
      cluster = cfg->attrs[i].val.clusterDim.x * cfg->attrs[i].val.clusterDim.y * cfg->attrs[i].val.clusterDim.z;
  const long long key = 1 + ((long long)cluster << 1) +
                        ((long long)(cfg->blockDim.x * cfg->blockDim.y * cfg->blockDim.z) << 8) +
                        ((long long)cfg->dynamicSmemBytes << 20);
  unsigned long long ctx = current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_mu);
    const Entry* e = find(ctx, func, key);
    if (e) {
      *active = e->value;
      return cudaSuccess;
    }
  }
  int n = 0;
  const cudaError_t err = cudaOccupancyMaxActiveClusters(&n, func, cfg);
  if (err != cudaSuccess) return err;
  *active = n;
  if (ctx == 0) ctx = current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_mu);
    put(ctx, func, key, n);
  }
  return cudaSuccess;
}

}  // namespace specv
