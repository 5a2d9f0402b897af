// pack.cu -- one-time repacking of the layer's weights into the layout the GEMMs read.
//
//   W1  [L + 2 S Is, d]  rows 0..L-1: W_down; then the shared experts' gate and value rows
//                        interleaved in groups of 16 (16 gate rows of features f..f+15, then
//                        the 16 value rows of the same features), features ordered s*Is + i
//   Wr  [E, L]           router, unchanged
//   Wgu                  per expert, gate/value rows interleaved in groups of 16 likewise,
//                        stored as tiles (below)
//   Wed                  routed down-projections, stored as tiles (below)
//   (expert_fp8: Wgu and Wed hold e4m3 codes in tiles of 128 rows x 128 codes, the same
//   16 KB, plus one fp32 scale per row in Sgu / Sed; see quant.cu)
//   W2  [d, L + S Is]    row n = [ W_up[n, :] | W_sd[0][n, :] | ... | W_sd[S-1][n, :] ]
//   gamma [L] fp32
// Tiled expert weights: an expert's [M_w, Kd] matrix is cut into 128-row x 64-column tiles,
// ordered (expert, row tile, column tile), each stored as 128 consecutive rows of 64 bf16
// (16 KB, contiguous); rows past M_w in the last row tile are zero.  Every box the routed
// GEMMs load is then one contiguous 16 KB read.
// The interleave lets one 32-column slice of a GEMM accumulator hold 16 gate and the 16
// matching value pre-activations, so SiTU-GLU is applied in the GEMM epilogue.  The two
// shared experts then form one GLU of width S*Is, and the shared down-projection is
// concatenated with the up-projection along the reduction dimension so that
// y = [z | hs] . W2^T is a single GEMM.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

enum PackJob : int { PACK_W1 = 0, PACK_W2 = 2 };

struct PackArgs {
  int job;
  int rows;         // destination rows
  int cols;         // destination columns (bf16 elements)
  __nv_bfloat16* dst;
  // sources
  const __nv_bfloat16* a;  // w_down / w_gate / w_up
  const __nv_bfloat16* g;  // w_sgate / w_gate
  const __nv_bfloat16* v;  // w_svalue / w_value
  const __nv_bfloat16* sd; // w_sdown
  int d, L, I, S, Is;
};

__device__ __forceinline__ void copy_row(__nv_bfloat16* dst, const __nv_bfloat16* src, int n) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* o = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < n / 8; i += blockDim.x) o[i] = __ldg(s + i);
}

__global__ void __launch_bounds__(256) pack_kernel(const PackArgs p) {
  for (int r = blockIdx.x; r < p.rows; r += gridDim.x) {
    __nv_bfloat16* drow = p.dst + static_cast<size_t>(r) * p.cols;
    if (p.job == PACK_W1) {
      if (r < p.L) {
        copy_row(drow, p.a + static_cast<size_t>(r) * p.d, p.d);
      } else {
        const int rr = r - p.L;
        const int grp = rr / (2 * GLU_GROUP), w = rr % (2 * GLU_GROUP);
        const int f = grp * GLU_GROUP + (w % GLU_GROUP);  // shared feature s*Is + i
        const __nv_bfloat16* src = (w < GLU_GROUP ? p.g : p.v) + static_cast<size_t>(f) * p.d;
        copy_row(drow, src, p.d);
      }
    } else {  // PACK_W2, row n of the output width d
      copy_row(drow, p.a + static_cast<size_t>(r) * p.L, p.L);
      for (int s = 0; s < p.S; ++s)
        copy_row(drow + p.L + static_cast<size_t>(s) * p.Is,
                 p.sd + (static_cast<size_t>(s) * p.d + r) * p.Is, p.Is);
    }
  }
}

// Tiled expert weights.  glu = 1: rows are the gate/value interleave of w_g / w_v
// ([E, M_w / 2, Kd] each); glu = 0: rows of w ([E, M_w, Kd]).  One thread per 16-byte chunk.
__global__ void __launch_bounds__(256)
pack_tiled_kernel(__nv_bfloat16* __restrict__ dst, const __nv_bfloat16* __restrict__ w,
                  const __nv_bfloat16* __restrict__ w_g, const __nv_bfloat16* __restrict__ w_v,
                  int glu, int E, int M_w, int Kd) {
  const int mt = (M_w + BLOCK_M - 1) / BLOCK_M, nk = Kd / BLOCK_K;
  const int64_t chunks = static_cast<int64_t>(E) * mt * nk * BLOCK_M * (BLOCK_K / 8);
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = c >> 3;  // 8 chunks of 16 B per 64-column row
    const int ch = static_cast<int>(c & 7);
    const int r = static_cast<int>(row % BLOCK_M);
    const int64_t tile = row / BLOCK_M;
    const int kb = static_cast<int>(tile % nk);
    const int64_t em = tile / nk;
    const int m = static_cast<int>(em % mt);
    const int e = static_cast<int>(em / mt);
    const int lr = m * BLOCK_M + r;  // row within the expert
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (lr < M_w) {
      const __nv_bfloat16* src;
      if (glu) {
        const int grp = lr / (2 * GLU_GROUP), wi = lr % (2 * GLU_GROUP);
        const int f = grp * GLU_GROUP + (wi % GLU_GROUP);
        src = (wi < GLU_GROUP ? w_g : w_v) + (static_cast<size_t>(e) * (M_w / 2) + f) * Kd;
      } else {
        src = w + (static_cast<size_t>(e) * M_w + lr) * Kd;
      }
      val = __ldg(reinterpret_cast<const uint4*>(src + kb * BLOCK_K) + ch);
    }
    reinterpret_cast<uint4*>(dst)[c] = val;
  }
}

// Transposed tiled expert weights for the backward pass, same tile order as above.
// glu = 1: per expert [M_w = L rows, Kd = 2I cols], col k is packed gate/value row k
// (interleave of w_g / w_v [E, Kd/2, M_w]), element (r, k) = W_{g|v}[e][f(k)][r];
// glu = 0: per expert [M_w = I rows, Kd = L cols], element (r, k) = w[e][k][r] (w [E, Kd, M_w]).
__global__ void __launch_bounds__(256)
pack_tiled_t_kernel(__nv_bfloat16* __restrict__ dst, const __nv_bfloat16* __restrict__ w,
                    const __nv_bfloat16* __restrict__ w_g, const __nv_bfloat16* __restrict__ w_v,
                    int glu, int E, int M_w, int Kd) {
  const int mt = (M_w + BLOCK_M - 1) / BLOCK_M, nk = Kd / BLOCK_K;
  const int64_t chunks = static_cast<int64_t>(E) * mt * nk * BLOCK_M * (BLOCK_K / 8);
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = c >> 3;
    const int ch = static_cast<int>(c & 7);
    const int rr = static_cast<int>(row % BLOCK_M);
    const int64_t tile = row / BLOCK_M;
    const int kb = static_cast<int>(tile % nk);
    const int64_t em = tile / nk;
    const int m = static_cast<int>(em % mt);
    const int e = static_cast<int>(em / mt);
    const int r = m * BLOCK_M + rr;
    __nv_bfloat16 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = kb * BLOCK_K + ch * 8 + i;
      __nv_bfloat16 x = __float2bfloat16_rn(0.0f);
      if (r < M_w) {
        if (glu) {
          const int grp = k / (2 * GLU_GROUP), wi = k % (2 * GLU_GROUP);
          const int f = grp * GLU_GROUP + (wi % GLU_GROUP);
          x = (wi < GLU_GROUP ? w_g : w_v)[(static_cast<size_t>(e) * (Kd / 2) + f) * M_w + r];
        } else {
          x = w[(static_cast<size_t>(e) * Kd + k) * M_w + r];
        }
      }
      v[i] = x;
    }
    reinterpret_cast<uint4*>(dst)[c] = *reinterpret_cast<const uint4*>(v);
  }
}

int launch_pack_backward(const lmoe_dims& D, const lmoe_weights& w, __nv_bfloat16* wgu_t,
                         __nv_bfloat16* wed_t, cudaStream_t stream) {
  pack_tiled_t_kernel<<<8192, 256, 0, stream>>>(wgu_t, nullptr,
                                                static_cast<const __nv_bfloat16*>(w.w_gate),
                                                static_cast<const __nv_bfloat16*>(w.w_value), 1,
                                                D.E, D.L, 2 * D.I);
  if (cudaGetLastError() != cudaSuccess) return LMOE_ERR_CUDA;
  pack_tiled_t_kernel<<<8192, 256, 0, stream>>>(wed_t, static_cast<const __nv_bfloat16*>(w.w_edown),
                                                nullptr, nullptr, 0, D.E, D.I, D.L);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

static int run_pack_tiled(__nv_bfloat16* dst, const __nv_bfloat16* w, const __nv_bfloat16* w_g,
                          const __nv_bfloat16* w_v, int glu, int E, int M_w, int Kd,
                          cudaStream_t stream) {
  pack_tiled_kernel<<<4096, 256, 0, stream>>>(dst, w, w_g, w_v, glu, E, M_w, Kd);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

static int run_pack(const PackArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return LMOE_OK;
  const int grid = a.rows < 4096 ? a.rows : 4096;
  pack_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

int launch_pack(const lmoe_dims& D, const lmoe_weights& w, const PackedLayout& P, uint8_t* base,
                cudaStream_t stream) {
  using bf = __nv_bfloat16;
  PackArgs a{};
  a.d = D.d;
  a.L = D.L;
  a.I = D.I;
  a.S = D.S;
  a.Is = D.Is;
  int rc;

  a.job = PACK_W1;
  a.rows = D.L + 2 * D.S * D.Is;
  a.cols = D.d;
  a.dst = reinterpret_cast<bf*>(base + P.w1);
  a.a = static_cast<const bf*>(w.w_down);
  a.g = static_cast<const bf*>(w.w_sgate);
  a.v = static_cast<const bf*>(w.w_svalue);
  if ((rc = run_pack(a, stream)) != LMOE_OK) return rc;

  if (D.expert_fp8) {
    if ((rc = launch_pack_tiled_e4m3(base + P.wgu, reinterpret_cast<float*>(base + P.sgu),
                                     nullptr, static_cast<const bf*>(w.w_gate),
                                     static_cast<const bf*>(w.w_value), 1, D.E, 2 * D.I, D.L,
                                     stream)) != LMOE_OK)
      return rc;
    if ((rc = launch_pack_tiled_e4m3(base + P.wed, reinterpret_cast<float*>(base + P.sed),
                                     static_cast<const bf*>(w.w_edown), nullptr, nullptr, 0, D.E,
                                     D.L, D.I, stream)) != LMOE_OK)
      return rc;
  } else {
    if ((rc = run_pack_tiled(reinterpret_cast<bf*>(base + P.wgu), nullptr,
                             static_cast<const bf*>(w.w_gate), static_cast<const bf*>(w.w_value),
                             1, D.E, 2 * D.I, D.L, stream)) != LMOE_OK)
      return rc;
    if ((rc = run_pack_tiled(reinterpret_cast<bf*>(base + P.wed),
                             static_cast<const bf*>(w.w_edown), nullptr, nullptr, 0, D.E, D.L,
                             D.I, stream)) != LMOE_OK)
      return rc;
  }

  a.job = PACK_W2;
  a.rows = D.d;
  a.cols = D.L + D.S * D.Is;
  a.dst = reinterpret_cast<bf*>(base + P.w2);
  a.a = static_cast<const bf*>(w.w_up);
  a.sd = static_cast<const bf*>(w.w_sdown);
  if ((rc = run_pack(a, stream)) != LMOE_OK) return rc;

  if (cudaMemcpyAsync(base + P.wr, w.w_router, static_cast<size_t>(D.E) * D.L * 2,
                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (cudaMemcpyAsync(base + P.gamma, w.gamma, static_cast<size_t>(D.L) * 4,
                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

}  // namespace lmoe
