// stats.cu -- thresholds that persist across steps, and load statistics over steps.
//
// "Part 1 of Inside Kimi K3" (Towards AI article, Quantile Balancing passage): the routing
// thresholds are read off the distribution of the router scores at each step, and the point
// of balancing is that no expert sits idle while a few take the traffic.  Two step-to-step
// companions of the per-batch solve:
//   - streaming thresholds, the exponential moving average of the per-step thresholds,
//     fma(beta, tau_ema - tau_step, tau_step) in fp32 (tau_ema = tau_step on the first step);
//   - 64-bit load counters accumulated from each step's per-expert token counts.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

__global__ void __launch_bounds__(256)
tau_ema_kernel(const float* __restrict__ tau_step, float* __restrict__ tau_ema, int E,
               float beta, int first) {
  pdl_wait();
  pdl_launch_dependents();
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    const float s = tau_step[e];
    tau_ema[e] = first ? s : __fmaf_rn(beta, __fsub_rn(tau_ema[e], s), s);
  }
}

int launch_tau_ema(const float* tau_step, float* tau_ema, int E, float beta, int first,
                   cudaStream_t stream) {
  if (E == 0) return LMOE_OK;
  const unsigned grid = static_cast<unsigned>(ceil_div(E, 256));
  return launch_pdl(tau_ema_kernel, grid, 256, 0, stream, tau_step, tau_ema, E, beta, first) ==
                 cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

// One CTA.  counts[e] (or, without counts, offsets[e + 1] - offsets[e]) -> acc, laid out as
// documented at lmoe_load_stats_update.
constexpr int STATS_THREADS = 1024;

__global__ void __launch_bounds__(STATS_THREADS)
load_stats_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets, int E,
                  unsigned long long* __restrict__ acc) {
  __shared__ unsigned long long wsum[STATS_THREADS / 32], wmax[STATS_THREADS / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long pairs = 0, mx = 0;
  for (int e = threadIdx.x; e < E; e += STATS_THREADS) {
    const int32_t ci = counts ? counts[e] : offsets[e + 1] - offsets[e];
    const unsigned long long c = static_cast<unsigned long long>(ci < 0 ? 0 : ci);
    pairs += c;
    mx = c > mx ? c : mx;
    acc[4 + e] += c;
    acc[4 + E + e] += c * c;
    acc[4 + 2 * E + e] += c == 0 ? 1ull : 0ull;
    if (c > acc[4 + 3 * E + e]) acc[4 + 3 * E + e] = c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
    const unsigned long long m = __shfl_xor_sync(0xffffffffu, mx, o);
    mx = m > mx ? m : mx;
  }
  if (lane == 0) {
    wsum[warp] = pairs;
    wmax[warp] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long p = 0, m = 0;
    for (int w = 0; w < STATS_THREADS / 32; ++w) {
      p += wsum[w];
      m = wmax[w] > m ? wmax[w] : m;
    }
    acc[0] += 1;
    acc[1] += p;
    acc[2] += m;
    if (m > acc[3]) acc[3] = m;
  }
}

int launch_load_stats(const int32_t* counts, const int32_t* offsets, int E,
                      unsigned long long* acc, cudaStream_t stream) {
  return launch_pdl(load_stats_kernel, 1, STATS_THREADS, 0, stream, counts, offsets, E, acc) ==
                 cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

}  // namespace lmoe
