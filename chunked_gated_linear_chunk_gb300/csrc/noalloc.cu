// noalloc.cu -- gla_bwd_noalloc: the GLA backward with its scratch in a
// fixed device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the backward:
// a host framework that owns all device memory and gives its plugins no
// allocator, or a latency-critical training loop that forbids allocation
// after start-up.  They still own q, k, v, g, do and every output; only the
// scratch (gate-gradient partials, the final-state gate term and, with
// segment_ids, the document tables) comes from the array below.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds kNoAllocScratchBytes of it until the process exits.  In
// host code its name is only a host-side stand-in, so its device address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) and passed on like any workspace pointer.
#include <atomic>

#include "internal.cuh"

namespace glacore {

// Largest scratch the no-allocation backward can use (48 MiB).
constexpr size_t kNoAllocScratchBytes = GLACORE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device; the first call
// on each device does the lookup.
// The cache entries are atomics: host threads may race on the first lookup
// (they store the same address).
static glacore_status noalloc_scratch(void **out) {
  static std::atomic<void *> cache[128];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return GLACORE_ERR_CUDA;
  void *p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GLACORE_ERR_CUDA;
    cache[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return GLACORE_OK;
}

}  // namespace glacore

extern "C" glacore_status gla_bwd_noalloc(const glacore_problem *p, const void *do_,
                                          const float *dht, void *dq, void *dk, void *dv,
                                          float *dg, float *dh0, glacore_stream_t stream) {
  using namespace glacore;
  if (!p) return GLACORE_ERR_INVALID_ARG;
  glacore_problem q = *p;
  q.workspace = nullptr;
  q.workspace_bytes = 0;
  const size_t need = gla_bwd_workspace_size(&q);
  if (need > kNoAllocScratchBytes) return GLACORE_ERR_WORKSPACE;
  if (need > 0) {
    void *ws = nullptr;
    const glacore_status s = noalloc_scratch(&ws);
    if (s != GLACORE_OK) return s;
    q.workspace = ws;
    q.workspace_bytes = kNoAllocScratchBytes;
  }
  return gla_bwd(&q, do_, dht, dq, dk, dv, dg, dh0, stream);
}
