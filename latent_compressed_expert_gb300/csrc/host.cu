// host.cu -- lmoe_forward_host: the layer on batches in host memory, with each batch's copies
// overlapped with its neighbours' compute through caller-owned staging slots, streams and
// events (the library allocates nothing and creates nothing).
#include "common.cuh"
#include "kernels.cuh"

extern "C" int lmoe_forward_host(const lmoe_dims* dims, const void* packed, const void* x_host,
                                 int residual_is_x, void* y_host, void* workspace,
                                 size_t ws_bytes, lmoe_io* io, lmoe_host_pipe* pipe) {
  using namespace lmoe;
  if (io) io->kernel_launches = 0;
  if (!pipe || !dims) return LMOE_ERR_INVALID_ARG;
  // invalid or unsupported dims: lmoe_forward reports which, before it enqueues anything
  if (lmoe_workspace_bytes(dims) == 0)
    return lmoe_forward(dims, packed, nullptr, nullptr, nullptr, workspace, ws_bytes, io,
                        nullptr);
  const lmoe_dims& D = *dims;
  if (pipe->depth < 1 || pipe->depth > LMOE_HOST_PIPE_MAX_DEPTH || D.T > pipe->max_tokens)
    return LMOE_ERR_INVALID_ARG;
  if (D.T == 0) return LMOE_OK;
  if (!x_host || !y_host || !packed || !workspace || !pipe->upload || !pipe->compute ||
      !pipe->download)
    return LMOE_ERR_INVALID_ARG;
  const int k = static_cast<int>(pipe->calls % static_cast<unsigned long long>(pipe->depth));
  void* xd = pipe->x_dev[k];
  void* yd = pipe->y_dev[k];
  cudaEvent_t up_ev = static_cast<cudaEvent_t>(pipe->uploaded[k]);
  cudaEvent_t comp_ev = static_cast<cudaEvent_t>(pipe->computed[k]);
  cudaEvent_t down_ev = static_cast<cudaEvent_t>(pipe->downloaded[k]);
  if (!xd || !yd || !up_ev || !comp_ev || !down_ev) return LMOE_ERR_INVALID_ARG;
  // every check lmoe_forward makes, before the upload is enqueued
  const int chk = forward_args_check(dims, packed, xd, residual_is_x ? xd : nullptr, yd,
                                     workspace, ws_bytes, io);
  if (chk != LMOE_OK) return chk;
  cudaStream_t up = static_cast<cudaStream_t>(pipe->upload);
  cudaStream_t comp = static_cast<cudaStream_t>(pipe->compute);
  cudaStream_t down = static_cast<cudaStream_t>(pipe->download);
  const size_t bytes = static_cast<size_t>(D.T) * D.d * 2;
  if (pipe->calls >= static_cast<unsigned long long>(pipe->depth)) {
    // slot k was used before: its x buffer is free once that forward has run, its y buffer
    // once that download has run
    if (cudaStreamWaitEvent(up, comp_ev, 0) != cudaSuccess ||
        cudaStreamWaitEvent(comp, down_ev, 0) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  if (cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, up) != cudaSuccess ||
      cudaEventRecord(up_ev, up) != cudaSuccess || cudaStreamWaitEvent(comp, up_ev, 0) != cudaSuccess)
    return LMOE_ERR_CUDA;
  const int rc = lmoe_forward(dims, packed, xd, residual_is_x ? xd : nullptr, yd, workspace,
                              ws_bytes, io, comp);
  if (rc != LMOE_OK) return rc;
  if (cudaEventRecord(comp_ev, comp) != cudaSuccess ||
      cudaStreamWaitEvent(down, comp_ev, 0) != cudaSuccess ||
      cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, down) != cudaSuccess ||
      cudaEventRecord(down_ev, down) != cudaSuccess)
    return LMOE_ERR_CUDA;
  pipe->calls += 1;
  return LMOE_OK;
}
