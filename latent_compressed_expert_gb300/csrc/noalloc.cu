// noalloc.cu -- lmoe_forward_noalloc: the whole layer for small batches, with its scratch
// memory in a fixed array that lives in this library's device image instead of a workspace
// the caller allocates.
//
// Some callers cannot allocate device memory when they run the layer: plug-ins hosted by a
// framework that owns every device allocation through its own pool and hands extensions no
// raw memory; latency-critical serving loops where cudaMalloc/cudaFree would synchronise
// the device and stall other streams; deployments whose memory budget is fixed when the
// process starts.  This entry point lets them run a decode-sized batch with nothing but
// their inputs, outputs and the packed weights.
//
// The array below is reserved on every GPU on which this library's device code is loaded,
// for the life of the process.  Host code cannot use the array's name as a device address
// (in host code it names a host-side stand-in), so the device address is looked up with
// cudaGetSymbolAddress.  The runtime loads this library's device code into each CUDA context
// separately -- a second context on the same device, or the new primary context after
// cudaDeviceReset, holds its own copy of the array at its own address -- so the address is
// cached per context, keyed by the context's unique id (cuCtxGetId), which the driver never
// hands out twice in a process.  Without those driver calls it is looked up at every call.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t{24} << 20;
static_assert(NOALLOC_SCRATCH_BYTES == LMOE_NOALLOC_SCRATCH_BYTES, "header and library agree");

static __device__ __align__(256) uint8_t noalloc_scratch[NOALLOC_SCRATCH_BYTES];

typedef CUresult (*ctx_get_current_fn)(CUcontext*);
typedef CUresult (*ctx_get_id_fn)(CUcontext, unsigned long long*);

struct ContextApi {
  ctx_get_current_fn get_current = nullptr;
  ctx_get_id_fn get_id = nullptr;
};

static const ContextApi& context_api() {
  static ContextApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      api.get_current = reinterpret_cast<ctx_get_current_fn>(p);
    p = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      api.get_id = reinterpret_cast<ctx_get_id_fn>(p);
  });
  return api;
}

// Unique id of the context current on this thread; false if there is none or it cannot be read.
static bool current_context_id(unsigned long long* id) {
  const ContextApi& api = context_api();
  if (!api.get_current || !api.get_id) return false;
  CUcontext ctx = nullptr;
  if (api.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return api.get_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int NOALLOC_CACHE = 64;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
static ScratchEntry noalloc_cache[NOALLOC_CACHE];
static int noalloc_cached = 0;  // entries filled (a ring once all are)
static std::mutex noalloc_mutex;

// Device address of the array in the current context.  The first call in a context looks it
// up (which may load this library's device code into the context); later calls in the same
// context take it from the cache.
static int noalloc_scratch_for_current_context(void** out) {
  std::lock_guard<std::mutex> lock(noalloc_mutex);
  unsigned long long id = 0;
  if (current_context_id(&id)) {
    const int n = noalloc_cached < NOALLOC_CACHE ? noalloc_cached : NOALLOC_CACHE;
    for (int i = 0; i < n; ++i) {
      if (noalloc_cache[i].ctx_id == id) {
        *out = noalloc_cache[i].addr;
        return LMOE_OK;
      }
    }
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) return LMOE_ERR_CUDA;
  // the lookup makes the device's primary context current if no context was: key by the
  // context it resolved in
  if (current_context_id(&id)) {
    noalloc_cache[noalloc_cached % NOALLOC_CACHE] = ScratchEntry{id, p};
    ++noalloc_cached;
  }
  *out = p;
  return LMOE_OK;
}

}  // namespace lmoe

extern "C" int lmoe_forward_noalloc(const lmoe_dims* dims, const void* packed, const void* x,
                                    const void* residual, void* y, lmoe_io* io, void* stream) {
  using namespace lmoe;
  // invalid or unsupported dims: lmoe_forward reports which, before it enqueues anything
  if (lmoe_workspace_bytes(dims) == 0)
    return lmoe_forward(dims, packed, x, residual, y, nullptr, 0, io, stream);
  // the array must hold the base workspace; a small batch's split-K region is used when the
  // array also has room for it
  const size_t need = workspace_layout(*dims).total_base;
  if (need > NOALLOC_SCRATCH_BYTES) return LMOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int rc = noalloc_scratch_for_current_context(&scratch);
  if (rc != LMOE_OK) return rc;
  // lmoe_forward zeroes the one word that must start at zero (the device error flag) and
  // writes every other scratch buffer before reading it.
  return lmoe_forward(dims, packed, x, residual, y, scratch, NOALLOC_SCRATCH_BYTES, io, stream);
}

extern "C" int lmoe_noalloc_last_device_error(void) {
  using namespace lmoe;
  void* scratch = nullptr;
  const int rc = noalloc_scratch_for_current_context(&scratch);
  if (rc != LMOE_OK) return rc;
  // the array's first word is the forward workspace's device error flag
  return lmoe_last_device_error(scratch);
}
