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

// Tile shape of every GEMM: 128 rows (UMMA M) x BLOCK_N columns x 64 (one 128-byte
// swizzle atom of bf16 along K).
constexpr int BLOCK_M = 128;
constexpr int BLOCK_K = 64;
// Gate/value rows are interleaved in groups of 16 so that one 32-column TMEM load holds
// 16 gate and the matching 16 value accumulators of the same row.
constexpr int GLU_GROUP = 16;

// Tokens per block in the dispatch (permute) kernels: one 32-bit mask word per expert.
constexpr int DISPATCH_TOKENS = 32;

// Largest token count (MMA N) of one routed-expert GEMM tile; an expert's token rows are cut
// into chunks of at most this many.  192 covers the K3 prefill load (146 on average, under
// 1.2x that at most with Quantile-Balancing thresholds) in one chunk.
#ifndef LMOE_GROUPED_TOKN
#define LMOE_GROUPED_TOKN 192
#endif
constexpr int GROUPED_TOKN = LMOE_GROUPED_TOKN;

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

}  // namespace lmoe
