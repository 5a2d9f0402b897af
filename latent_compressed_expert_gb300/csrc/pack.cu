// pack.cu -- one-time repacking of the layer's weights into the layout the GEMMs read.
//
//   W1  [L + 2 S Is, d]  rows 0..L-1: W_down; then the shared experts' gate and value rows
//                        interleaved in groups of 16 (16 gate rows of features f..f+15, then
//                        the 16 value rows of the same features), features ordered s*Is + i
//   Wr  [E, L]           router, unchanged
//   Wgu [E, 2 I, L]      per expert, gate/value rows interleaved in groups of 16 likewise
//   Wed [E, L, I]        routed down-projections, unchanged
//   W2  [d, L + S Is]    row n = [ W_up[n, :] | W_sd[0][n, :] | ... | W_sd[S-1][n, :] ]
//   gamma [L] fp32
// The interleave lets one 32-column slice of a GEMM accumulator hold 16 gate and the 16
// matching value pre-activations, so SiTU-GLU is applied in the GEMM epilogue.  The two
// shared experts then form one GLU of width S*Is, and the shared down-projection is
// concatenated with the up-projection along the reduction dimension so that
// y = [z | hs] . W2^T is a single GEMM.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

enum PackJob : int { PACK_W1 = 0, PACK_WGU = 1, PACK_W2 = 2 };

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
    } else if (p.job == PACK_WGU) {
      const int e = r / (2 * p.I), rr = r % (2 * p.I);
      const int grp = rr / (2 * GLU_GROUP), w = rr % (2 * GLU_GROUP);
      const int f = grp * GLU_GROUP + (w % GLU_GROUP);
      const __nv_bfloat16* src =
          (w < GLU_GROUP ? p.g : p.v) + (static_cast<size_t>(e) * p.I + f) * p.L;
      copy_row(drow, src, p.L);
    } else {  // PACK_W2, row n of the output width d
      copy_row(drow, p.a + static_cast<size_t>(r) * p.L, p.L);
      for (int s = 0; s < p.S; ++s)
        copy_row(drow + p.L + static_cast<size_t>(s) * p.Is,
                 p.sd + (static_cast<size_t>(s) * p.d + r) * p.Is, p.Is);
    }
  }
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

  a.job = PACK_WGU;
  a.rows = D.E * 2 * D.I;
  a.cols = D.L;
  a.dst = reinterpret_cast<bf*>(base + P.wgu);
  a.g = static_cast<const bf*>(w.w_gate);
  a.v = static_cast<const bf*>(w.w_value);
  if ((rc = run_pack(a, stream)) != LMOE_OK) return rc;

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
  if (cudaMemcpyAsync(base + P.wed, w.w_edown, static_cast<size_t>(D.E) * D.L * D.I * 2,
                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (cudaMemcpyAsync(base + P.gamma, w.gamma, static_cast<size_t>(D.L) * 4,
                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

}  // namespace lmoe
