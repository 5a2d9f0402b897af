// bwd.cu -- backward pass of the routed-expert branch (element-wise and layout kernels).
//
// "Part 1 of Inside Kimi K3" (Towards AI article, stabilizers passage): SiTU-GLU and the
// RMSNorm after expert aggregation were introduced to keep training of the routed branch
// stable.  For the branch  h = SiTU(lat W_g^T, lat W_v^T),  o = h W_ed^T,  u = sum_j g_j o_j,
// z = gamma u r  with  r = (mean(u^2) + eps)^-1/2,  and an incoming dz:
//   a = gamma * dz,   du = r a - u r^3 <u, a> / L,   dgamma = sum_t dz u r,
//   do_j = g_j du,    dg_j = <du, o_j>,
//   dh -> through SiTU: with G = c tanh(g/c), V = c tanh(v/c), s = sigmoid(G):
//     dg_pre = dh V s (1 + G (1 - s)) (1 - (G/c)^2),   dv_pre = dh G s (1 - (V/c)^2),
// and the GEMMs (dgrad on transposed expert weights, wgrad as per-expert reductions over the
// expert's tokens) run in gemm_grouped.cu / gemm.cu.  Routing is a discrete choice and is
// held fixed.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace lmoe {

constexpr int BWD_MAX_VEC = 4;
constexpr int BWD_THREADS = 512;

__device__ __forceinline__ void bf8_to_f(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 f_to_bf8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Block-wide sum of one value per thread, in a fixed tree (warps, then warp 0).
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    float x = lane < nw ? red[lane] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red[32] = x;
  }
  __syncthreads();
  return red[32];
}

// One CTA per token: u and r exactly as the forward's combine computed them (fp32 fma in
// slot order, the same tree for the sum of squares), then du, do_j (bf16, at the permuted
// row of (t, j)) and dg_j; u and r are kept for dgamma.  STAGED: the token's K expert-output
// rows are first copied into shared memory (bulk copies on one mbarrier, a bounded wait;
// on time-out the CTA records the error bit and writes nothing), and both passes over them
// read shared memory; else both read global memory.
constexpr int BWD_BULK_MAX = 114688;  // bytes of staged rows per CTA (16 x 3584 bf16)

template <bool STAGED, int VEC>  // VEC: 8-feature vectors per thread
__global__ void __launch_bounds__(BWD_THREADS)
combine_bwd_kernel(const __nv_bfloat16* __restrict__ o, const float* __restrict__ gate,
                   const int32_t* __restrict__ inv, const float* __restrict__ gamma,
                   const float* __restrict__ dz, int K, int L, float eps,
                   __nv_bfloat16* __restrict__ dout, float* __restrict__ dgate,
                   float* __restrict__ u_out, float* __restrict__ r_out,
                   uint32_t* __restrict__ err, unsigned long long timeout_ns) {
  extern __shared__ __align__(128) uint8_t cbw_smem[];
  __shared__ int32_t rows[32];
  __shared__ float gates[32];
  __shared__ float red[33];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int t = blockIdx.x;
  if (STAGED && threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t row_bytes = static_cast<uint32_t>(L) * 2;
  if (threadIdx.x < K) {
    rows[threadIdx.x] = __ldg(inv + static_cast<size_t>(t) * K + threadIdx.x);
    gates[threadIdx.x] = __ldg(gate + static_cast<size_t>(t) * K + threadIdx.x);
  }
  __syncthreads();
  if (STAGED && threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(&bar, row_bytes * static_cast<uint32_t>(K));
    for (int j = 0; j < K; ++j)
      ptx::bulk_load(cbw_smem + static_cast<size_t>(j) * row_bytes,
                     o + static_cast<size_t>(rows[j]) * L, row_bytes, &bar);
  }
  const int nvec = L / 8;
  // slot j's 8-feature vector v
  auto orow = [&](int j, int v) -> uint4 {
    if constexpr (STAGED)
      return reinterpret_cast<const uint4*>(cbw_smem)[static_cast<size_t>(j) * nvec + v];
    else
      return __ldg(reinterpret_cast<const uint4*>(o + static_cast<size_t>(rows[j]) * L) + v);
  };
  if constexpr (STAGED) {
    const bool ok = ptx::mbar_wait(&bar, 0u, &abort_flag, timeout_ns);
    if (!__syncthreads_and(ok ? 1 : 0)) {
      if (threadIdx.x == 0) atomicOr(err, DEVERR_TIMEOUT_EPILOGUE);
      // copies still in flight must land before the CTA exits (bounded again)
      ptx::mbar_wait(&bar, 0u, &abort_flag, timeout_ns);
      return;
    }
  }
  float u[VEC][8];
  float ss = 0.0f;
#pragma unroll
  for (int c = 0; c < VEC; ++c) {
    const int v = threadIdx.x + c * blockDim.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) u[c][i] = 0.0f;
    if (v < nvec) {
      for (int j = 0; j < K; ++j) {
        float f[8];
        bf8_to_f(orow(j, v), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) u[c][i] = fmaf(gates[j], f[i], u[c][i]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(u[c][i], u[c][i], ss);
    }
  }
  const float r = rsqrtf(block_sum(ss, red) / static_cast<float>(L) + eps);
  // <u, gamma dz>
  float ua = 0.0f;
  float a[VEC][8];
#pragma unroll
  for (int c = 0; c < VEC; ++c) {
    const int v = threadIdx.x + c * blockDim.x;
    if (v < nvec) {
      const float4* dzp = reinterpret_cast<const float4*>(dz + static_cast<size_t>(t) * L) + 2 * v;
      const float4* gp = reinterpret_cast<const float4*>(gamma) + 2 * v;
      const float4 d0 = __ldg(dzp), d1 = __ldg(dzp + 1), g0 = __ldg(gp), g1 = __ldg(gp + 1);
      const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
      const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a[c][i] = gg[i] * dd[i];
        ua = fmaf(u[c][i], a[c][i], ua);
      }
      float4* up = reinterpret_cast<float4*>(u_out + static_cast<size_t>(t) * L) + 2 * v;
      up[0] = make_float4(u[c][0], u[c][1], u[c][2], u[c][3]);
      up[1] = make_float4(u[c][4], u[c][5], u[c][6], u[c][7]);
    }
  }
  const float coef = block_sum(ua, red) * r * r * r / static_cast<float>(L);
  if (threadIdx.x == 0) r_out[t] = r;
  // du, then do_j = g_j du and the per-thread parts of dg_j = <du, o_j>
  float dg[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) dg[j] = 0.0f;
#pragma unroll
  for (int c = 0; c < VEC; ++c) {
    const int v = threadIdx.x + c * blockDim.x;
    if (v < nvec) {
      float du[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) du[i] = r * a[c][i] - u[c][i] * coef;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < K) {
          float f[8], d[8];
          bf8_to_f(orow(j, v), f);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            d[i] = gates[j] * du[i];
            dg[j] = fmaf(du[i], f[i], dg[j]);
          }
          reinterpret_cast<uint4*>(dout + static_cast<size_t>(rows[j]) * L)[v] = f_to_bf8(d);
        }
      }
    }
  }
  // dg_j: warp sums, then one fixed-order sum over the warps (in the dynamic buffer, which
  // the staged rows no longer need: 2 CTAs of 112 KB rows fit an SM)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float (*dgs)[33] = reinterpret_cast<float (*)[33]>(cbw_smem);
  if constexpr (STAGED) __syncthreads();
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float x = dg[j];
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    if (lane == 0) dgs[warp][j] = x;
  }
  __syncthreads();
  if (threadIdx.x < K) {
    float s = 0.0f;
    for (int w = 0; w < static_cast<int>((blockDim.x + 31) >> 5); ++w) s += dgs[w][threadIdx.x];
    dgate[static_cast<size_t>(t) * K + threadIdx.x] = s;
  }
}

// dgamma[l] = sum_t dz[t, l] u[t, l] r[t], in two fixed-order passes: BWD_CHUNKS row chunks,
// then the chunks.
constexpr int BWD_CHUNKS = 64;

__global__ void __launch_bounds__(256)
colsum_kernel(const float* __restrict__ dz, const float* __restrict__ u,
              const float* __restrict__ r, int T, int L, float* __restrict__ part) {
  pdl_wait();
  pdl_launch_dependents();
  const int l = blockIdx.x * blockDim.x + threadIdx.x;
  const int chunk = blockIdx.y;
  if (l >= L) return;
  const int per = (T + BWD_CHUNKS - 1) / BWD_CHUNKS;
  const int t0 = chunk * per, t1 = min(T, t0 + per);
  float s = 0.0f;
  for (int t = t0; t < t1; ++t) {
    const size_t i = static_cast<size_t>(t) * L + l;
    s = fmaf(__ldg(dz + i) * __ldg(u + i), __ldg(r + t), s);
  }
  part[static_cast<size_t>(chunk) * L + l] = s;
}

__global__ void __launch_bounds__(256)
colsum_final_kernel(const float* __restrict__ part, int L, float* __restrict__ dgamma) {
  pdl_wait();
  pdl_launch_dependents();
  const int l = blockIdx.x * blockDim.x + threadIdx.x;
  if (l >= L) return;
  float s = 0.0f;
  for (int c = 0; c < BWD_CHUNKS; ++c) s += part[static_cast<size_t>(c) * L + l];
  dgamma[l] = s;
}

// SiTU-GLU backward on the interleaved gate/value layout: row p of pre / dgv holds, for each
// group of GLU_GROUP features, GLU_GROUP gate then GLU_GROUP value pre-activations.  A thread
// takes 8 consecutive features of one row: 16-byte loads of their gate, value and dh, and
// 16-byte stores of both gradients.  tanh and the exponential are the hardware approximations
// (relative error about 2^-11, below the bf16 rounding of the operands and of the result).
__global__ void __launch_bounds__(256)
situ_bwd_kernel(const __nv_bfloat16* __restrict__ pre, const __nv_bfloat16* __restrict__ dh,
                int64_t rows, int I, float c, __nv_bfloat16* __restrict__ dgv, int64_t ldo) {
  pdl_wait();
  pdl_launch_dependents();
  const int per_row = I / 8;
  const int64_t n = rows * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = i / per_row;
    const int f = static_cast<int>(i - p * per_row) * 8;  // first feature
    const int col = (f / GLU_GROUP) * 2 * GLU_GROUP + f % GLU_GROUP;  // its gate column
    float g[8], v[8], d[8], dg[8], dv[8];
    bf8_to_f(__ldg(reinterpret_cast<const uint4*>(pre + p * 2 * I + col)), g);
    bf8_to_f(__ldg(reinterpret_cast<const uint4*>(pre + p * 2 * I + col + GLU_GROUP)), v);
    bf8_to_f(__ldg(reinterpret_cast<const uint4*>(dh + p * I + f)), d);
    const float inv_c = 1.0f / c;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float tg = ptx::tanh_approx(g[k] * inv_c), tv = ptx::tanh_approx(v[k] * inv_c);
      const float G = c * tg, V = c * tv;
      const float sg = __fdividef(1.0f, 1.0f + __expf(fminf(-G, 80.0f)));
      dg[k] = d[k] * V * sg * (1.0f + G * (1.0f - sg)) * (1.0f - tg * tg);
      dv[k] = d[k] * G * sg * (1.0f - tv * tv);
    }
    *reinterpret_cast<uint4*>(dgv + p * ldo + col) = f_to_bf8(dg);
    *reinterpret_cast<uint4*>(dgv + p * ldo + col + GLU_GROUP) = f_to_bf8(dv);
  }
}

// dlat[t] = add[t] + sum_j x[inv[t, j]] in slot order (fp32; add optional), and optionally
// its bf16 copy into row t of outb (row stride ldb).
__global__ void __launch_bounds__(BWD_THREADS)
slot_sum_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ inv, int K,
                int L, const float* __restrict__ add, float* __restrict__ out,
                __nv_bfloat16* __restrict__ outb, int64_t ldb) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int nvec = L / 8;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (add) {
      const float4* a4 = reinterpret_cast<const float4*>(add + static_cast<size_t>(t) * L) + 2 * v;
      const float4 a0 = __ldg(a4), a1 = __ldg(a4 + 1);
      acc[0] = a0.x; acc[1] = a0.y; acc[2] = a0.z; acc[3] = a0.w;
      acc[4] = a1.x; acc[5] = a1.y; acc[6] = a1.z; acc[7] = a1.w;
    }
    for (int j = 0; j < K; ++j) {
      float f[8];
      const int row = __ldg(inv + static_cast<size_t>(t) * K + j);
      bf8_to_f(__ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * L) + v), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
    float4* o = reinterpret_cast<float4*>(out + static_cast<size_t>(t) * L) + 2 * v;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if (outb) {
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(outb + static_cast<size_t>(t) * ldb + 8 * v) =
          make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

// XT[w, q] = x[q, w] for q < n, zero for n <= q < qmax (qmax = the grid's 64-row tiles):
// 64 x 64 tiles through shared memory, 16-byte row loads, and 16-byte stores of eight
// consecutive q of one output row (a warp reads 32 consecutive w of one tile row).
constexpr int TP_TILE = 64;
constexpr int TP_PITCH = TP_TILE + 8;  // bf16 per shared row; keeps 16-byte row stores aligned

__global__ void __launch_bounds__(256)
transpose_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx, int W, int64_t n,
                      int64_t ldt, __nv_bfloat16* __restrict__ xt) {
  __shared__ __align__(16) __nv_bfloat16 tile[TP_TILE][TP_PITCH];
  pdl_wait();
  pdl_launch_dependents();
  const int w0 = blockIdx.y * TP_TILE;
  const int64_t q0 = static_cast<int64_t>(blockIdx.x) * TP_TILE;
  const int c = threadIdx.x & 7;  // 16-byte chunk of a 64-wide row
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = (threadIdx.x >> 3) + 32 * i;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (q0 + r < n && w0 + 8 * c < W)
      v = __ldg(reinterpret_cast<const uint4*>(x + (q0 + r) * ldx + w0 + 8 * c));
    *reinterpret_cast<uint4*>(&tile[r][8 * c]) = v;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, qc = threadIdx.x >> 5;  // q chunk per warp
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int wl = lane + 32 * i;
    if (w0 + wl >= W) continue;
    uint32_t pk[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = __bfloat16_as_ushort(tile[8 * qc + 2 * j][wl]);
      const uint32_t hi = __bfloat16_as_ushort(tile[8 * qc + 2 * j + 1][wl]);
      pk[j] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(xt + static_cast<int64_t>(w0 + wl) * ldt + q0 + 8 * qc) =
        make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

// out[p, :W] = x[idx[p], :W] for p < n (16-byte pieces; W, ldx and ldo multiples of 8).  One
// warp per row; each lane issues all its loads of a row (up to GATHER_VEC 16-byte pieces)
// before their stores, and the stores stream (the rows are written once, while the source
// rows, re-read by every slot of their token, stay in L2).
constexpr int GATHER_WARPS = 8;
constexpr int GATHER_VEC = 16;  // 16-byte pieces per lane held at once: W <= 4096 in one pass

__global__ void __launch_bounds__(32 * GATHER_WARPS)
gather_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx,
                   const int32_t* __restrict__ idx, int64_t n, int W,
                   __nv_bfloat16* __restrict__ out, int64_t ldo) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t p = static_cast<int64_t>(blockIdx.x) * GATHER_WARPS + (threadIdx.x >> 5);
  if (p >= n) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(__ldg(idx + p)) * ldx);
  uint4* dst = reinterpret_cast<uint4*>(out + p * ldo);
  const int nv = W / 8;
  for (int v0 = 0; v0 < nv; v0 += GATHER_VEC * 32) {
    uint4 r[GATHER_VEC];
#pragma unroll
    for (int k = 0; k < GATHER_VEC; ++k) {
      const int v = v0 + k * 32 + lane;
      if (v < nv) r[k] = __ldg(src + v);
    }
#pragma unroll
    for (int k = 0; k < GATHER_VEC; ++k) {
      const int v = v0 + k * 32 + lane;
      if (v < nv) __stcs(dst + v, r[k]);
    }
  }
}

int launch_gather_rows(const __nv_bfloat16* x, int64_t ldx, const int32_t* idx, int64_t n, int W,
                       __nv_bfloat16* out, int64_t ldo, cudaStream_t stream) {
  if (n == 0) return LMOE_OK;
  if (W % 8 || ldx % 8 || ldo % 8 || (reinterpret_cast<uintptr_t>(x) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15) || ceil_div(n, GATHER_WARPS) > 0x7fffffff)
    return LMOE_ERR_UNSUPPORTED;
  return launch_pdl(gather_rows_kernel, static_cast<unsigned>(ceil_div(n, GATHER_WARPS)),
                    32 * GATHER_WARPS, 0, stream, x, ldx, idx, n, W, out, ldo) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

// Output row of each packed row: rows below `base` keep their place; the 2I gate/value rows
// after them (interleaved in groups of GLU_GROUP) go to base + f (gate feature f) and
// base + I + f (value feature f).  With `seg`, also writes the one-group range {0, seg_len}.
__global__ void rowmap_kernel(int I, int base, int32_t* __restrict__ map,
                              int32_t* __restrict__ seg, int seg_len) {
  const int i0 = blockIdx.x * blockDim.x + threadIdx.x;
  if (seg && i0 == 0) {
    seg[0] = 0;
    seg[1] = seg_len;
  }
  for (int k = i0; k < base + 2 * I; k += gridDim.x * blockDim.x) {
    if (k < base) {
      map[k] = k;
      continue;
    }
    const int kk = k - base;
    const int grp = kk / (2 * GLU_GROUP), wi = kk % (2 * GLU_GROUP);
    const int f = grp * GLU_GROUP + (wi % GLU_GROUP);
    map[k] = base + (wi < GLU_GROUP ? f : I + f);
  }
}

int launch_rowmap(int I, int base, int32_t* map, int32_t* seg, int seg_len, cudaStream_t stream) {
  const int n = base + 2 * I > 1 ? base + 2 * I : 1;
  rowmap_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, stream>>>(I, base, map, seg,
                                                                              seg_len);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

// ------------------------------------------------------------------------------------
int launch_combine_bwd(const __nv_bfloat16* o, const float* gate, const int32_t* inv,
                       const float* gamma, const float* dz, int T, int K, int L, float eps,
                       __nv_bfloat16* dout, float* dgate, float* u, float* r, uint32_t* err,
                       unsigned long long timeout_ns, cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  const int nvec = L / 8;
  const int threads = static_cast<int>(ceil_div(nvec < BWD_THREADS ? nvec : BWD_THREADS, 32) * 32);
  if (nvec > BWD_MAX_VEC * threads || K > 32) return LMOE_ERR_UNSUPPORTED;
  const size_t dgs_bytes = (BWD_THREADS / 32) * 33 * sizeof(float);
  const size_t staged = static_cast<size_t>(K) * L * 2;
  if (staged <= static_cast<size_t>(BWD_BULK_MAX) && nvec <= threads &&
      !(reinterpret_cast<uintptr_t>(o) & 15)) {
    // one vector per thread keeps the registers of two 112 KB CTAs within an SM's
    const size_t smem = staged > dgs_bytes ? staged : dgs_bytes;
    if (cudaFuncSetAttribute(combine_bwd_kernel<true, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LMOE_ERR_CUDA;
    return launch_pdl(combine_bwd_kernel<true, 1>, T, threads, smem, stream, o, gate, inv, gamma,
                      dz, K, L, eps, dout, dgate, u, r, err, timeout_ns) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  }
  return launch_pdl(combine_bwd_kernel<false, BWD_MAX_VEC>, T, threads, dgs_bytes, stream, o, gate,
                    inv, gamma, dz, K, L, eps, dout, dgate, u, r, err, timeout_ns) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_dgamma(const float* dz, const float* u, const float* r, int T, int L, float* part,
                  float* dgamma, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(ceil_div(L, 256)), BWD_CHUNKS);
  if (launch_pdl(colsum_kernel, grid, 256, 0, stream, dz, u, r, T, L, part) != cudaSuccess ||
      launch_pdl(colsum_final_kernel, static_cast<unsigned>(ceil_div(L, 256)), 256, 0, stream,
                 static_cast<const float*>(part), L, dgamma) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

int launch_situ_bwd(const __nv_bfloat16* pre, const __nv_bfloat16* dh, int64_t rows, int I,
                    float c, __nv_bfloat16* dgv, int64_t ldo, cudaStream_t stream) {
  if (rows == 0) return LMOE_OK;
  if (I % GLU_GROUP || ldo % 8 || (reinterpret_cast<uintptr_t>(pre) & 15) ||
      (reinterpret_cast<uintptr_t>(dh) & 15) || (reinterpret_cast<uintptr_t>(dgv) & 15))
    return LMOE_ERR_UNSUPPORTED;
  const int64_t n = rows * (I / 8);
  const unsigned grid = static_cast<unsigned>(ceil_div(n, 256) < 65535 * 16 ? ceil_div(n, 256) : 65535 * 16);
  return launch_pdl(situ_bwd_kernel, grid, 256, 0, stream, pre, dh, rows, I, c, dgv, ldo) ==
                 cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_slot_sum(const __nv_bfloat16* x, const int32_t* inv, int T, int K, int L,
                    const float* add, float* out, __nv_bfloat16* outb, int64_t ldb,
                    cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  if (outb && (ldb % 8 || (reinterpret_cast<uintptr_t>(outb) & 15))) return LMOE_ERR_UNSUPPORTED;
  return launch_pdl(slot_sum_kernel, T, BWD_THREADS, 0, stream, x, inv, K, L, add, out, outb,
                    ldb) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_transpose_rows(const __nv_bfloat16* x, int64_t ldx, int W, int64_t n, int64_t qmax,
                          int64_t ldt, __nv_bfloat16* xt, cudaStream_t stream) {
  if (n == 0 && qmax == 0) return LMOE_OK;
  // 16-byte rows and stores; whole 64-row tiles
  if (qmax < n || W % 8 || ldx % 8 || ldt % 8 || ldt < qmax || qmax % TP_TILE ||
      (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(xt) & 15))
    return LMOE_ERR_UNSUPPORTED;
  if (ceil_div(W, TP_TILE) > 65535) return LMOE_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(qmax / TP_TILE),
                  static_cast<unsigned>(ceil_div(W, TP_TILE)));
  return launch_pdl(transpose_rows_kernel, grid, 256, 0, stream, x, ldx, W, n, ldt, xt) ==
                 cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

}  // namespace lmoe
