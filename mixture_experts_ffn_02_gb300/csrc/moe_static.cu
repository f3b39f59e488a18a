// moe_route_static: top-k routing for callers that cannot allocate device
// memory.
//
// moe_route needs a workspace for its per-block partial counts and
// probability sums.  Some callers have no way to provide one: code that runs
// where cudaMalloc is forbidden or unavailable (inside a captured region of a
// host framework that owns every allocation, a custom allocator that hands
// out only the tensors it tracks, an embedded runtime with a fixed memory
// plan).  This entry point keeps that scratch in a fixed array that lives in
// the library's own device memory, so the caller passes only inputs and
// outputs.
//
// The array holds MOE_ROUTE_STATIC_SCRATCH_BYTES (512 KiB) per GPU that
// loads the library, for as long as the process lives.  All calls on a GPU
// share it, and it keeps whatever the last call left there: the one value
// that must start at zero (the last-block ticket counter) is cleared at the
// start of every call.  Calls whose kernels overlap on the same GPU (for
// example on two streams at once) race on the array and must not be issued.
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr size_t kStaticScratch = MOE_ROUTE_STATIC_SCRATCH_BYTES;

// The scratch itself.  Host code must not pass this name to a kernel: on the
// host it only stands in for the symbol; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_route_scratch[kStaticScratch];

// Device address of the scratch per device, cached once found.  A failed
// lookup is not cached: the next call on that device tries again.
std::mutex g_addr_mu;
void* g_addr[64] = {};

// Device address of the scratch on the current device (with that device
// current).  No allocation happens here.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();          // clear the error the failed query recorded
      return MOE_ERR_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_route_static(const moe_config* cfg, const moe_tensors* t, int* device_status,
                                void* stream) {
  int rc = moe_check_config(cfg);
  if (rc) return rc;
  if (!t) return MOE_ERR_NULL;
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return MOE_ERR_CUDA;
  if (di.cc_major != 10) return MOE_ERR_DEVICE;
  const void* need[] = {t->logits, t->topk_idx, t->gates, t->counts, t->f, t->p, t->aux};
  for (const void* q : need) {
    if (!q) return MOE_ERR_NULL;
    if (!aligned16(q)) return MOE_ERR_ALIGN;
  }
  if ((t->bias && !aligned16(t->bias)) || (t->valid && !aligned16(t->valid)))
    return MOE_ERR_ALIGN;
  // Same grid as moe_route, so both produce the same bytes.
  WsLayout w;
  ws_layout(cfg, 0, &w);
  // route totals (zeroed by the launch), then one int per route block
  const size_t need_bytes = kRouteAccBytes + (size_t)w.route_blocks * sizeof(int);
  if (need_bytes > kStaticScratch) return MOE_ERR_WORKSPACE;

  void* base = nullptr;
  if ((rc = scratch_address(&base))) return rc;
  char* sc = static_cast<char*>(base);
  int* treal = reinterpret_cast<int*>(sc + kRouteAccBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_route_scratch(*cfg, t->logits, t->bias, t->valid, t->topk_idx, t->gates,
                           t->counts, t->f, t->p, t->aux, sc, treal, device_status,
                           w.route_blocks, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
