// dispatch.cu -- token dispatch into expert-contiguous segments (indices only: the routed
// gate/value GEMM gathers the latent rows itself), and the gate-weighted aggregation fused
// with RMSNorm.
//
// Sources: "The 2.8-Trillion-Parameter Problem: Why Bigger Models Break the Old Playbook"
// ("Part 1 of Inside Kimi K3", Towards AI article): each selected expert receives the
// token's (latent) vector, works on it, and the outputs are combined and projected back
// up; an RMSNorm sits right before the up-projection.  "苏神复盘 Kimi K3" ("Merged
// summary", Stable LatentMoE bullet): RMSNorm after expert aggregation and before the
// up-projection normalises the branch scale.
//
// Dispatch is deterministic: within an expert's segment, rows are in token order.  A block
// of 32 tokens records, per expert, a 32-bit mask of the tokens that picked it; a token's
// rank inside the segment is the number of earlier blocks' picks (a column prefix sum)
// plus the popcount of the lower mask bits.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

// masks[b][e] bit i <=> token 32 b + i selected expert e.
__global__ void __launch_bounds__(256)
dispatch_mask_kernel(const int32_t* __restrict__ idx, int T, int E, int K,
                     uint32_t* __restrict__ masks, uint32_t* __restrict__ err) {
  extern __shared__ uint32_t m_smem[];
  const int b = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) m_smem[e] = 0u;
  __syncthreads();
  const int t0 = b * DISPATCH_TOKENS;
  const int ntok = min(DISPATCH_TOKENS, T - t0);
  for (int p = threadIdx.x; p < ntok * K; p += blockDim.x) {
    const int tl = p / K;
    const int e = __ldg(idx + static_cast<size_t>(t0) * K + p);
    if (e < 0 || e >= E) {
      atomicOr(err, DEVERR_BAD_INDEX);
      continue;
    }
    atomicOr(&m_smem[e], 1u << tl);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    masks[static_cast<size_t>(b) * E + e] = m_smem[e];
}

// One CTA: base[b][e] = picks of expert e in blocks < b; offsets = exclusive scan of the
// counts over experts; ct_off = exclusive scan of ceil(count / GROUPED_TOKN) (the token
// chunks of the routed-expert GEMMs).
__global__ void __launch_bounds__(1024)
dispatch_scan_kernel(const uint32_t* __restrict__ masks, int nb, int E, int TK,
                     uint32_t* __restrict__ base, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ ct_off, int32_t* __restrict__ counts_out) {
  __shared__ int32_t warp_cnt[32], warp_mt[32];
  __shared__ int32_t carry_cnt, carry_mt;
  if (threadIdx.x == 0) {
    carry_cnt = 0;
    carry_mt = 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    int cnt = 0;
    if (e < E) {
      int b = 0;
      for (; b + 4 <= nb; b += 4) {
        const uint32_t m0 = __ldg(masks + static_cast<size_t>(b) * E + e);
        const uint32_t m1 = __ldg(masks + static_cast<size_t>(b + 1) * E + e);
        const uint32_t m2 = __ldg(masks + static_cast<size_t>(b + 2) * E + e);
        const uint32_t m3 = __ldg(masks + static_cast<size_t>(b + 3) * E + e);
        base[static_cast<size_t>(b) * E + e] = cnt;
        cnt += __popc(m0);
        base[static_cast<size_t>(b + 1) * E + e] = cnt;
        cnt += __popc(m1);
        base[static_cast<size_t>(b + 2) * E + e] = cnt;
        cnt += __popc(m2);
        base[static_cast<size_t>(b + 3) * E + e] = cnt;
        cnt += __popc(m3);
      }
      for (; b < nb; ++b) {
        base[static_cast<size_t>(b) * E + e] = cnt;
        cnt += __popc(__ldg(masks + static_cast<size_t>(b) * E + e));
      }
      if (counts_out) counts_out[e] = cnt;
    }
    const int mt = static_cast<int>(ceil_div(cnt, GROUPED_TOKN));
    // block-wide exclusive scans of cnt and mt
    int ic = cnt, im = mt;
    for (int o = 1; o < 32; o <<= 1) {
      const int vc = __shfl_up_sync(0xffffffffu, ic, o);
      const int vm = __shfl_up_sync(0xffffffffu, im, o);
      if (lane >= o) {
        ic += vc;
        im += vm;
      }
    }
    if (lane == 31) {
      warp_cnt[warp] = ic;
      warp_mt[warp] = im;
    }
    __syncthreads();
    if (warp == 0) {
      const int nw = blockDim.x >> 5;
      int wc = lane < nw ? warp_cnt[lane] : 0, wm = lane < nw ? warp_mt[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int vc = __shfl_up_sync(0xffffffffu, wc, o);
        const int vm = __shfl_up_sync(0xffffffffu, wm, o);
        if (lane >= o) {
          wc += vc;
          wm += vm;
        }
      }
      if (lane < nw) {
        warp_cnt[lane] = wc;  // inclusive over warps
        warp_mt[lane] = wm;
      }
    }
    __syncthreads();
    const int before_c = (warp > 0 ? warp_cnt[warp - 1] : 0) + (ic - cnt);
    const int before_m = (warp > 0 ? warp_mt[warp - 1] : 0) + (im - mt);
    if (e < E) {
      offsets[e] = carry_cnt + before_c;
      ct_off[e] = carry_mt + before_m;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_cnt += warp_cnt[(blockDim.x >> 5) - 1];
      carry_mt += warp_mt[(blockDim.x >> 5) - 1];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    offsets[E] = carry_cnt;  // == T*K when every index was valid
    ct_off[E] = carry_mt;
    (void)TK;
  }
}

// Scatter: inv[t*K + j] = row of (t, j) in the permuted order, and src_tok[row] = t (the
// routed gate/value GEMM gathers the latent rows through it).  One thread per pair.
__global__ void __launch_bounds__(256)
dispatch_scatter_kernel(const int32_t* __restrict__ idx, const uint32_t* __restrict__ masks,
                        const uint32_t* __restrict__ base, const int32_t* __restrict__ offsets,
                        int T, int E, int K, int32_t* __restrict__ inv,
                        int32_t* __restrict__ src_tok) {
  const int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (p >= static_cast<int64_t>(T) * K) return;
  const int t = static_cast<int>(p / K);
  const int b = t / DISPATCH_TOKENS, tl = t % DISPATCH_TOKENS;
  const int e = __ldg(idx + p);
  if (e < 0 || e >= E) return;  // flagged by the mask kernel
  const size_t me = static_cast<size_t>(b) * E + e;
  const int row = __ldg(offsets + e) + static_cast<int>(__ldg(base + me)) +
                  __popc(__ldg(masks + me) & ((1u << tl) - 1u));
  inv[p] = row;
  src_tok[row] = t;
}

// Combine + RMSNorm: one CTA per token, each thread owns 8 consecutive latent features
// (a 16-byte vector), for up to COMBINE_MAX_VEC vectors (L <= 16384).  u accumulates the K expert rows in
// fp32 in slot order; the sum of squares is reduced in a fixed tree, so the result does not
// depend on scheduling.
constexpr int COMBINE_MAX_VEC = 4;
constexpr int COMBINE_MAX_THREADS = 512;
constexpr int COMBINE_BATCH = 4;  // row loads issued together

__global__ void __launch_bounds__(COMBINE_MAX_THREADS)
combine_rmsnorm_kernel(const __nv_bfloat16* __restrict__ o, const float* __restrict__ gate,
                       const int32_t* __restrict__ inv, const float* __restrict__ gamma,
                       int T, int K, int L, float eps, __nv_bfloat16* __restrict__ z,
                       int ldz) {
  __shared__ int32_t rows[32];
  __shared__ float gates[32];
  __shared__ float warp_ss[32];
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    rows[threadIdx.x] = __ldg(inv + static_cast<size_t>(t) * K + threadIdx.x);
    gates[threadIdx.x] = __ldg(gate + static_cast<size_t>(t) * K + threadIdx.x);
  }
  __syncthreads();
  const int nvec = L / 8;
  float u[COMBINE_MAX_VEC][8];
  float ss = 0.0f;
#pragma unroll
  for (int c = 0; c < COMBINE_MAX_VEC; ++c) {
    const int v = threadIdx.x + c * blockDim.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) u[c][i] = 0.0f;
    if (v < nvec) {
      // the loads of COMBINE_BATCH rows are issued before their sums, in slot order
      for (int j0 = 0; j0 < K; j0 += COMBINE_BATCH) {
        uint4 raw[COMBINE_BATCH];
#pragma unroll
        for (int jj = 0; jj < COMBINE_BATCH; ++jj)
          if (j0 + jj < K)
            raw[jj] = __ldg(reinterpret_cast<const uint4*>(o + static_cast<size_t>(rows[j0 + jj]) * L) + v);
#pragma unroll
        for (int jj = 0; jj < COMBINE_BATCH; ++jj) {
          if (j0 + jj < K) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[jj]);
            const float g = gates[j0 + jj];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __bfloat1622float2(h[i]);
              u[c][2 * i] = fmaf(g, f.x, u[c][2 * i]);
              u[c][2 * i + 1] = fmaf(g, f.y, u[c][2 * i + 1]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(u[c][i], u[c][i], ss);
    }
  }
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_ss[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    float v = lane < nw ? warp_ss[lane] : 0.0f;
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) warp_ss[0] = v;
  }
  __syncthreads();
  const float inv_rms = rsqrtf(warp_ss[0] / static_cast<float>(L) + eps);
#pragma unroll
  for (int c = 0; c < COMBINE_MAX_VEC; ++c) {
    const int v = threadIdx.x + c * blockDim.x;
    if (v < nvec) {
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v);
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v + 1);
      const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      uint4 out;
      __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ob[i] = __floats2bfloat162_rn(u[c][2 * i] * inv_rms * gm[2 * i],
                                      u[c][2 * i + 1] * inv_rms * gm[2 * i + 1]);
      reinterpret_cast<uint4*>(z + static_cast<size_t>(t) * ldz)[v] = out;
    }
  }
}

// ------------------------------------------------------------------------------------
int launch_dispatch(const int32_t* idx, int T, int E, int K, uint32_t* masks, uint32_t* base,
                    int32_t* offsets, int32_t* ct_off, int32_t* inv, int32_t* src_tok,
                    int32_t* counts_out, uint32_t* err, cudaStream_t stream) {
  const int nb = static_cast<int>(ceil_div(T, DISPATCH_TOKENS));
  const size_t msmem = static_cast<size_t>(E) * sizeof(uint32_t);
  if (nb > 0) {
    dispatch_mask_kernel<<<nb, 256, msmem, stream>>>(idx, T, E, K, masks, err);
    if (cudaGetLastError() != cudaSuccess) return LMOE_ERR_CUDA;
  }
  dispatch_scan_kernel<<<1, 1024, 0, stream>>>(masks, nb, E, T * K, base, offsets, ct_off,
                                               counts_out);
  if (cudaGetLastError() != cudaSuccess) return LMOE_ERR_CUDA;
  if (nb > 0) {
    const int64_t pairs = static_cast<int64_t>(T) * K;
    dispatch_scatter_kernel<<<static_cast<unsigned>(ceil_div(pairs, 256)), 256, 0, stream>>>(
        idx, masks, base, offsets, T, E, K, inv, src_tok);
    if (cudaGetLastError() != cudaSuccess) return LMOE_ERR_CUDA;
  }
  return LMOE_OK;
}

int launch_combine(const __nv_bfloat16* o, const float* gate, const int32_t* inv,
                   const float* gamma, int T, int K, int L, float eps, __nv_bfloat16* z,
                   int ldz, cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  const int nvec = L / 8;
  const int threads = static_cast<int>(
      ceil_div(nvec < COMBINE_MAX_THREADS ? nvec : COMBINE_MAX_THREADS, 32) * 32);
  if (nvec > COMBINE_MAX_VEC * threads) return LMOE_ERR_UNSUPPORTED;
  combine_rmsnorm_kernel<<<T, threads, 0, stream>>>(o, gate, inv, gamma, T, K, L, eps, z, ldz);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

}  // namespace lmoe
