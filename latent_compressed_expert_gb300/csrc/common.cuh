// common.cuh -- shared definitions of the lmoe CUDA library (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lmoe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "lmoe is written for sm_103a only"
#endif

namespace lmoe {

// Device error flag bits (first word of the forward workspace).
constexpr uint32_t DEVERR_TIMEOUT_PRODUCER = 1u << 0;
constexpr uint32_t DEVERR_TIMEOUT_MMA = 1u << 1;
constexpr uint32_t DEVERR_TIMEOUT_EPILOGUE = 1u << 2;
constexpr uint32_t DEVERR_TIMEOUT_DRAIN = 1u << 3;
constexpr uint32_t DEVERR_BAD_INDEX = 1u << 8;
constexpr uint32_t DEVERR_NONFINITE = 1u << 9;  // checked mode: a non-finite router logit

// Tile shape of every GEMM: 128 rows (UMMA M) x BLOCK_N columns x 64 (one 128-byte
// swizzle atom of bf16 along K).
constexpr int BLOCK_M = 128;
constexpr int BLOCK_K = 64;
// Gate/value rows are interleaved in groups of 16 so that one 32-column TMEM load holds
// 16 gate and the matching 16 value accumulators of the same row.
constexpr int GLU_GROUP = 16;

// Tokens per block in the dispatch (permute) kernels: one 32-bit mask word per expert.
constexpr int DISPATCH_TOKENS = 32;

// Token chunks of the routed-expert GEMMs (MMA N): an expert's token rows are cut into
// ceil(count / tokn) chunks of equal size (to one row), tokn = GROUPED_TOKN or, when experts
// average more than that, GROUPED_TOKN_WIDE.  192 covers the K3 prefill load (146 on average,
// under 1.2x that at most with Quantile-Balancing thresholds) in one chunk; at 585 tokens per
// expert (T = 32768) 256 makes three chunks of 195 instead of four.
constexpr int GROUPED_TOKN = 192;
constexpr int GROUPED_TOKN_WIDE = 256;
constexpr int GROUPED_TOKN_NARROW = 128;  // the e4m3 down GEMM's chunks (see grouped_tokn_down)

// The chunk size of a batch, a function of its dims only, so that the forward and the
// backward, which reads the forward's chunk offsets, agree.
inline int grouped_tokn(int64_t T, int K, int E) {
  return E > 0 && T * K / E > GROUPED_TOKN ? GROUPED_TOKN_WIDE : GROUPED_TOKN;
}

// The forward's bf16 gate/value GEMM takes GROUPED_TOKN chunks whatever the batch's are (a
// second prefix sum when they differ): with ~585 tokens per expert that made it 3.40 -> 3.30 ms,
// while the down GEMM runs faster on the wider chunks.  The e4m3 gate/value GEMM (single weight
// tiles) keeps the batch's chunks: 2.13 ms on them against 2.30 ms on GROUPED_TOKN ones.
inline int grouped_tokn_gate_up(int64_t T, int K, int E, bool fp8) {
  return fp8 ? grouped_tokn(T, K, E) : GROUPED_TOKN;
}

// The forward's e4m3 down GEMM at decode-like loads (fewer than 32 tokens per expert on
// average) takes 128-token chunks (a second prefix sum when the batch's differ), so that its
// weight-tile pairs' accumulators (2 x 128 columns) fit TMEM twice and its drain overlaps the
// next tile's MMAs: 0.180 -> 0.164 ms at T = 64.  At 146 tokens per expert the split chunks
// cost more than the overlap gains (0.577 -> 0.606 ms).
inline int grouped_tokn_down(int64_t T, int K, int E, bool fp8) {
  return fp8 && E > 0 && T * K / E < 32 ? GROUPED_TOKN_NARROW : grouped_tokn(T, K, E);
}

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Programmatic dependent launch.  Every kernel of the forward is launched with
// launch_pdl: the GPU may start it while the previous kernel of the stream is still
// finishing.  Each kernel first does the set-up that touches no global memory (barrier
// init, TMEM allocation, tensor-map prefetch), then pdl_wait(), which returns once the
// previous grid has completed and its writes are visible -- so every global access keeps
// stream order -- and then pdl_launch_dependents(), which lets the next kernel start its own
// set-up.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}


__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

}  // namespace lmoe
