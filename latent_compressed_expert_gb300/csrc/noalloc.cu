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
// cudaGetSymbolAddress once per device, on the first call made with that device current,
// and cached.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t{24} << 20;
static_assert(NOALLOC_SCRATCH_BYTES == LMOE_NOALLOC_SCRATCH_BYTES, "header and library agree");

static __device__ __align__(256) uint8_t noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
static void* noalloc_scratch_addr[NOALLOC_MAX_DEVICES];
static std::mutex noalloc_mutex;

// Device address of the array on the current device (looked up once per device).
static int noalloc_scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMOE_ERR_CUDA;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return LMOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(noalloc_mutex);
  if (noalloc_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return LMOE_ERR_CUDA;
    noalloc_scratch_addr[dev] = p;
  }
  *out = noalloc_scratch_addr[dev];
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
  const int rc = noalloc_scratch_for_current_device(&scratch);
  if (rc != LMOE_OK) return rc;
  // lmoe_forward zeroes the one word that must start at zero (the device error flag) and
  // writes every other scratch buffer before reading it.
  return lmoe_forward(dims, packed, x, residual, y, scratch, NOALLOC_SCRATCH_BYTES, io, stream);
}
