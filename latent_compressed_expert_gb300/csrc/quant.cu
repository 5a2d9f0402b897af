// quant.cu -- e4m3 (FP8) quantisation of the routed experts' GEMM operands.
//
// "苏神复盘 Kimi K3" ("Merged summary", Stable LatentMoE bullet): SiTU-GLU soft-caps the
// outliers that would otherwise blow up the BF16/FP8 dynamic range, i.e. the routed branch
// is meant to run in FP8.  The pages give no recipe; the one used here: each row (one
// output feature of one expert's weight matrix, or one activation row) gets one fp32 scale
// s = amax / 448 (1 when that is 0), and its values become e4m3(x / s), rounded to nearest
// even and saturating at 448, every step an IEEE fp32 operation.  The GEMM multiplies its
// fp32 sum by both rows' scales.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace lmoe {

constexpr float E4M3_MAX = 448.0f;
constexpr int QUANT_WARPS = 8;

__device__ __forceinline__ void bf16x8_to_float(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// 16 values -> 16 codes (byte i = code of value i).
__device__ __forceinline__ uint4 quantize16(const float (&f)[16], float s) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t lo = ptx::cvt_e4m3x2(__fdiv_rn(f[4 * i + 1], s), __fdiv_rn(f[4 * i], s));
    const uint16_t hi = ptx::cvt_e4m3x2(__fdiv_rn(f[4 * i + 3], s), __fdiv_rn(f[4 * i + 2], s));
    w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float row_scale(float amax) {
  const float s = __fdiv_rn(amax, E4M3_MAX);
  return s > 0.0f ? s : 1.0f;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp per row of `cols` bf16 values (cols % 16 == 0): codes [rows, ldq], scales [rows].
// Rows of 2..QUANT_HOLD chunks of 16 values per lane are held in registers (one read of the
// row, every load issued before the reduction); other rows are read twice.
constexpr int QUANT_HOLD = 8;

__global__ void __launch_bounds__(QUANT_WARPS * 32)
quantize_rows_held_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int cols,
                          int64_t ldx, uint8_t* __restrict__ q, int64_t ldq,
                          float* __restrict__ scales) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * QUANT_WARPS + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + r * ldx);
  const int nch = cols / 16;
  uint4 hold[2 * QUANT_HOLD];
#pragma unroll
  for (int i = 0; i < QUANT_HOLD; ++i) {
    const int c = lane + 32 * i;
    if (c < nch) {
      hold[2 * i] = __ldg(xr + 2 * c);
      hold[2 * i + 1] = __ldg(xr + 2 * c + 1);
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < QUANT_HOLD; ++i) {
    if (lane + 32 * i < nch) {
      float f[8];
      bf16x8_to_float(hold[2 * i], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
      bf16x8_to_float(hold[2 * i + 1], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
    }
  }
  const float s = row_scale(warp_max(amax));
  uint4* qr = reinterpret_cast<uint4*>(q + r * ldq);
#pragma unroll
  for (int i = 0; i < QUANT_HOLD; ++i) {
    const int c = lane + 32 * i;
    if (c < nch) {
      float f[16], a[8];
      bf16x8_to_float(hold[2 * i], a);
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] = a[k];
      bf16x8_to_float(hold[2 * i + 1], a);
#pragma unroll
      for (int k = 0; k < 8; ++k) f[8 + k] = a[k];
      qr[c] = quantize16(f, s);
    }
  }
  if (lane == 0) scales[r] = s;
}

__global__ void __launch_bounds__(QUANT_WARPS * 32)
quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
                     uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scales) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * QUANT_WARPS + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + r * ldx);  // 8 values per uint4
  const int nch = cols / 16;
  float amax = 0.0f;
  for (int c = lane; c < nch; c += 32) {
    float f[8];
    bf16x8_to_float(__ldg(xr + 2 * c), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    bf16x8_to_float(__ldg(xr + 2 * c + 1), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  const float s = row_scale(warp_max(amax));
  uint4* qr = reinterpret_cast<uint4*>(q + r * ldq);
  for (int c = lane; c < nch; c += 32) {
    float f[16], a[8];
    bf16x8_to_float(__ldg(xr + 2 * c), a);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = a[i];
    bf16x8_to_float(__ldg(xr + 2 * c + 1), a);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[8 + i] = a[i];
    qr[c] = quantize16(f, s);
  }
  if (lane == 0) scales[r] = s;
}

int launch_quantize_rows(const __nv_bfloat16* x, int64_t rows, int cols, int64_t ldx,
                         uint8_t* q, int64_t ldq, float* scales, cudaStream_t stream) {
  if (rows == 0) return LMOE_OK;
  if (cols <= 0 || cols % 16 || ldx % 8 || ldq % 16) return LMOE_ERR_UNSUPPORTED;
  const int64_t grid = ceil_div(rows, QUANT_WARPS);
  // the held kernel pays for its registers only when a lane holds several chunks (measured:
  // 3584-wide latent rows gain, 512-wide SiTU rows lose occupancy)
  if (cols > 32 * 16 && cols <= 32 * 16 * QUANT_HOLD)
    return launch_pdl(quantize_rows_held_kernel, static_cast<unsigned>(grid), QUANT_WARPS * 32, 0,
                      stream, x, rows, cols, ldx, q, ldq, scales) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  return launch_pdl(quantize_rows_kernel, static_cast<unsigned>(grid), QUANT_WARPS * 32, 0, stream,
                    x, rows, cols, ldx, q, ldq, scales) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

// Expert weights -> e4m3 tiles of 128 rows x 128 codes (16 KB, ordered (expert, row tile,
// column tile), like the bf16 tiles) and one scale per row ([E * mt * 128]; padding rows of
// the last row tile get code 0 and scale 0).  glu = 1: the rows are the gate/value
// interleave of w_g / w_v (groups of GLU_GROUP rows); glu = 0: the rows of w.  One warp per
// packed row.
__global__ void __launch_bounds__(QUANT_WARPS * 32)
pack_tiled_e4m3_kernel(uint8_t* __restrict__ dst, float* __restrict__ scales,
                       const __nv_bfloat16* __restrict__ w, const __nv_bfloat16* __restrict__ w_g,
                       const __nv_bfloat16* __restrict__ w_v, int glu, int E, int M_w, int Kd) {
  const int lane = threadIdx.x & 31;
  const int mt = (M_w + BLOCK_M - 1) / BLOCK_M;
  const int nk = Kd / 128;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * QUANT_WARPS + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(E) * mt * BLOCK_M) return;
  const int e = static_cast<int>(row / (static_cast<int64_t>(mt) * BLOCK_M));
  const int lr = static_cast<int>(row % (static_cast<int64_t>(mt) * BLOCK_M));  // in expert
  const int m = lr / BLOCK_M, rr = lr % BLOCK_M;
  const bool valid = lr < M_w;
  const __nv_bfloat16* src = nullptr;
  if (valid) {
    if (glu) {
      const int grp = lr / (2 * GLU_GROUP), wi = lr % (2 * GLU_GROUP);
      const int f = grp * GLU_GROUP + (wi % GLU_GROUP);
      src = (wi < GLU_GROUP ? w_g : w_v) + (static_cast<size_t>(e) * (M_w / 2) + f) * Kd;
    } else {
      src = w + (static_cast<size_t>(e) * M_w + lr) * Kd;
    }
  }
  const uint4* sr = reinterpret_cast<const uint4*>(src);
  const int nch = Kd / 16;
  float amax = 0.0f;
  if (valid) {
    for (int c = lane; c < nch; c += 32) {
      float f[8];
      bf16x8_to_float(__ldg(sr + 2 * c), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
      bf16x8_to_float(__ldg(sr + 2 * c + 1), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    }
  }
  const float s = row_scale(warp_max(amax));
  const size_t tile0 = (static_cast<size_t>(e) * mt + m) * nk;
  for (int c = lane; c < nch; c += 32) {
    const int k0 = c * 16;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
      float f[16], a[8];
      bf16x8_to_float(__ldg(sr + 2 * c), a);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = a[i];
      bf16x8_to_float(__ldg(sr + 2 * c + 1), a);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[8 + i] = a[i];
      out = quantize16(f, s);
    }
    uint8_t* d = dst + (tile0 + k0 / 128) * (BLOCK_M * 128) + static_cast<size_t>(rr) * 128 +
                 (k0 % 128);
    *reinterpret_cast<uint4*>(d) = out;
  }
  if (lane == 0) scales[row] = valid ? s : 0.0f;
}

int launch_pack_tiled_e4m3(uint8_t* dst, float* scales, const __nv_bfloat16* w,
                           const __nv_bfloat16* w_g, const __nv_bfloat16* w_v, int glu, int E,
                           int M_w, int Kd, cudaStream_t stream) {
  if (Kd % 128) return LMOE_ERR_UNSUPPORTED;
  const int64_t rows = static_cast<int64_t>(E) * ceil_div(M_w, BLOCK_M) * BLOCK_M;
  pack_tiled_e4m3_kernel<<<static_cast<unsigned>(ceil_div(rows, QUANT_WARPS)), QUANT_WARPS * 32,
                           0, stream>>>(dst, scales, w, w_g, w_v, glu, E, M_w, Kd);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

}  // namespace lmoe
