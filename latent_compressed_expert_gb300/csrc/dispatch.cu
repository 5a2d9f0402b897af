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
#include "ptx.cuh"

namespace lmoe {

// masks[b][e] bit i <=> token 32 b + i selected expert e.
__global__ void __launch_bounds__(256)
dispatch_mask_kernel(const int32_t* __restrict__ idx, int T, int E, int K,
                     uint32_t* __restrict__ masks, uint32_t* __restrict__ err,
                     uint32_t* __restrict__ done) {
  extern __shared__ uint32_t m_smem[];
  const int b = blockIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  if (b == 0 && threadIdx.x == 0) *done = 0u;  // completion counter of the column scan
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

// Column scan: base[b][e] = picks of expert e in blocks < b, and the expert's count.  A CTA
// owns 32 experts (one per lane, so every mask row is read as one 128-byte line); its 16 warps
// split the blocks into strips: each thread sums its strip, the strips' sums are scanned
// across the warps, and a second pass over the strip writes the bases.  The counts go to
// offsets[e]; the last CTA to finish (a fence and an atomic counter that the mask kernel
// zeroed, no waiting) turns them into the exclusive scans offsets (rows) and ct_off (token
// chunks of the routed-expert GEMMs, ceil(count / tokn)).
constexpr int SCAN_WARPS = 16;
constexpr int SCAN_THREADS = SCAN_WARPS * 32;

__global__ void __launch_bounds__(SCAN_THREADS)
dispatch_scan_kernel(const uint32_t* __restrict__ masks, int nb, int E,
                     uint32_t* __restrict__ base, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ ct_off, int tokn, int32_t* __restrict__ ct_off2,
                     int tokn2, int32_t* __restrict__ counts_out, uint32_t* __restrict__ done) {
  __shared__ uint32_t part[SCAN_WARPS][32];
  __shared__ int32_t wsum[3][SCAN_WARPS];
  __shared__ bool last;
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int per = (nb + SCAN_WARPS - 1) / SCAN_WARPS;
  const int b0 = warp * per, b1 = min(nb, b0 + per);
  uint32_t sum = 0u;
  if (e < E) {
#pragma unroll 4
    for (int b = b0; b < b1; ++b) sum += __popc(__ldg(masks + static_cast<size_t>(b) * E + e));
  }
  part[warp][lane] = sum;
  __syncthreads();
  uint32_t run = 0u, total = 0u;
  for (int w = 0; w < SCAN_WARPS; ++w) {
    const uint32_t v = part[w][lane];
    run += w < warp ? v : 0u;
    total += v;
  }
  if (e < E) {
    for (int b = b0; b < b1; ++b) {
      const size_t me = static_cast<size_t>(b) * E + e;
      base[me] = run;
      run += __popc(__ldg(masks + me));
    }
    if (warp == 0) {
      offsets[e] = static_cast<int32_t>(total);
      if (counts_out) counts_out[e] = static_cast<int32_t>(total);
    }
  }
  // the last CTA scans the counts of all experts
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int eper = (E + SCAN_THREADS - 1) / SCAN_THREADS;
  const int e0 = threadIdx.x * eper, e1 = min(E, e0 + eper);
  const bool two = ct_off2 != nullptr;
  int32_t c_rows = 0, c_chunks = 0, c_chunks2 = 0;
  for (int i = e0; i < e1; ++i) {
    const int32_t c = __ldcg(offsets + i);
    c_rows += c;
    c_chunks += static_cast<int32_t>(ceil_div(c, tokn));
    if (two) c_chunks2 += static_cast<int32_t>(ceil_div(c, tokn2));
  }
  int32_t ir = c_rows, ic = c_chunks, ic2 = c_chunks2;  // inclusive scans within the warp
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t vr = __shfl_up_sync(0xffffffffu, ir, o);
    const int32_t vc = __shfl_up_sync(0xffffffffu, ic, o);
    const int32_t vc2 = __shfl_up_sync(0xffffffffu, ic2, o);
    if (lane >= o) {
      ir += vr;
      ic += vc;
      ic2 += vc2;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = ir;
    wsum[1][warp] = ic;
    wsum[2][warp] = ic2;
  }
  __syncthreads();
  int32_t pr = ir - c_rows, pc = ic - c_chunks, pc2 = ic2 - c_chunks2;
  int32_t tr = 0, tc = 0, tc2 = 0;
  for (int w = 0; w < SCAN_WARPS; ++w) {
    pr += w < warp ? wsum[0][w] : 0;
    pc += w < warp ? wsum[1][w] : 0;
    pc2 += w < warp ? wsum[2][w] : 0;
    tr += wsum[0][w];
    tc += wsum[1][w];
    tc2 += wsum[2][w];
  }
  // every count was read above: the exclusive scans overwrite them in place
  __syncthreads();
  for (int i = e0; i < e1; ++i) {
    const int32_t c = __ldcg(offsets + i);
    offsets[i] = pr;
    ct_off[i] = pc;
    pr += c;
    pc += static_cast<int32_t>(ceil_div(c, tokn));
    if (two) {
      ct_off2[i] = pc2;
      pc2 += static_cast<int32_t>(ceil_div(c, tokn2));
    }
  }
  if (threadIdx.x == 0) {
    offsets[E] = tr;  // == T*K when every index was valid
    ct_off[E] = tc;
    if (two) ct_off2[E] = tc2;
  }
}

// Scatter: inv[t*K + j] = row of (t, j) in the permuted order, and src_tok[row] = t (the
// routed gate/value GEMM gathers the latent rows through it).  One thread per pair.
__global__ void __launch_bounds__(256)
dispatch_scatter_kernel(const int32_t* __restrict__ idx, const uint32_t* __restrict__ masks,
                        const uint32_t* __restrict__ base, const int32_t* __restrict__ offsets,
                        int T, int E, int K, int32_t* __restrict__ inv,
                        int32_t* __restrict__ src_tok) {
  pdl_wait();
  pdl_launch_dependents();
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
  pdl_wait();
  pdl_launch_dependents();
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

// u += gate_j rows[j] for the K staged rows j = 0..K-1, in that order (fp32 fused multiply-adds):
// thread i owns the 8-feature vectors i, i + blockDim.x, ... of the token.
__device__ __forceinline__ void combine_accumulate(const uint4* rows, const float* gates, int K,
                                                   int L, float (&u)[COMBINE_MAX_VEC][8]) {
  const int nvec = L / 8;
#pragma unroll
  for (int c = 0; c < COMBINE_MAX_VEC; ++c) {
    const int v = threadIdx.x + c * blockDim.x;
    if (v < nvec) {
      for (int j = 0; j < K; ++j) {
        const uint4 raw = rows[static_cast<size_t>(j) * nvec + v];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
        const float g = gates[j];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(h[i]);
          u[c][2 * i] = fmaf(g, f.x, u[c][2 * i]);
          u[c][2 * i + 1] = fmaf(g, f.y, u[c][2 * i + 1]);
        }
      }
    }
  }
}

// z = gamma * u / sqrt(mean(u^2) + eps): the sum of squares of each thread's vectors, then a
// fixed tree (lanes, then warps).  Called by every thread of the CTA (it synchronises).
__device__ __forceinline__ void combine_finish(const float (&u)[COMBINE_MAX_VEC][8],
                                               float* warp_ss, const float* gamma, int L,
                                               float eps, __nv_bfloat16* zrow) {
  const int nvec = L / 8;
  float ss = 0.0f;
#pragma unroll
  for (int c = 0; c < COMBINE_MAX_VEC; ++c) {
    const int v = threadIdx.x + c * blockDim.x;
    if (v < nvec) {
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
      reinterpret_cast<uint4*>(zrow)[v] = out;
    }
  }
}

// The same normalisation for threads that hold two vectors (v and v + blockDim.x, blockDim.x a
// multiple of 32), with the reduction tree of the one-vector-per-thread kernels above: vector v
// is summed as lane v % 32 of warp v / 32 whichever thread holds it, and the final tree runs
// over the same ceil(nvec / 32) warp sums.  So z has their bits, for any L up to 32 warps.
__device__ __forceinline__ void combine_finish_pairs(const float (&u)[COMBINE_MAX_VEC][8],
                                                     float* warp_ss, const float* gamma, int L,
                                                     float eps, __nv_bfloat16* zrow) {
  const int nvec = L / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwp = static_cast<int>(blockDim.x >> 5);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int v = threadIdx.x + c * blockDim.x;
    float ss = 0.0f;
    if (v < nvec) {
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(u[c][i], u[c][i], ss);
    }
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) warp_ss[warp + c * nwp] = ss;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = (nvec + 31) >> 5;
    float v = lane < nw ? warp_ss[lane] : 0.0f;
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) warp_ss[0] = v;
  }
  __syncthreads();
  const float inv_rms = rsqrtf(warp_ss[0] / static_cast<float>(L) + eps);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
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
      reinterpret_cast<uint4*>(zrow)[v] = out;
    }
  }
}

// The token's K expert rows staged in shared memory, in rounds of `rpp` rows (all K at once
// when rpp >= K): u accumulates in registers over the rounds in slot order, so a round size
// changes the footprint, not the arithmetic.
__device__ __forceinline__ void combine_staged_rows(const uint4* rows, const float* gates,
                                                    float* warp_ss, const float* gamma, int K,
                                                    int L, float eps, __nv_bfloat16* zrow) {
  float u[COMBINE_MAX_VEC][8];
#pragma unroll
  for (int c = 0; c < COMBINE_MAX_VEC; ++c)
#pragma unroll
    for (int i = 0; i < 8; ++i) u[c][i] = 0.0f;
  combine_accumulate(rows, gates, K, L, u);
  combine_finish(u, warp_ss, gamma, L, eps, zrow);
}

// Combine + RMSNorm with the token's K expert rows staged in shared memory by 1-D bulk
// copies: one thread issues the K copies on one mbarrier, so a CTA has all K rows in
// flight at once (K * L * 2 bytes; two CTAs per SM when that is at most COMBINE_BULK_MAX).
// Then each thread sums its 8-feature vectors over the slots in slot order, the sum of
// squares is reduced in the same fixed tree as above, and z is written.  The wait on the
// copies is bounded; on time-out the CTA records the error bit and writes nothing.
constexpr int COMBINE_BULK_MAX = 114688;  // bytes of staged rows per CTA (16 x 3584 bf16)
constexpr int COMBINE_ROUND_ROWS = 7;      // rows per round of combine_rounds_kernel (0: off)
__global__ void __launch_bounds__(COMBINE_MAX_THREADS)
combine_bulk_kernel(const __nv_bfloat16* __restrict__ o, const float* __restrict__ gate,
                    const int32_t* __restrict__ inv, const float* __restrict__ gamma, int T,
                    int K, int L, float eps, __nv_bfloat16* __restrict__ z, int ldz,
                    uint32_t* __restrict__ err, unsigned long long timeout_ns) {
  extern __shared__ __align__(128) uint8_t cb_smem[];
  __shared__ float gates[32];
  __shared__ float warp_ss[32];
  __shared__ __align__(8) uint64_t bar;
  const int t = blockIdx.x;
  const uint32_t row_bytes = static_cast<uint32_t>(L) * 2;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(&bar, row_bytes * static_cast<uint32_t>(K));
    for (int j = 0; j < K; ++j) {
      const int row = __ldg(inv + static_cast<size_t>(t) * K + j);
      ptx::bulk_load(cb_smem + static_cast<size_t>(j) * row_bytes,
                     o + static_cast<size_t>(row) * L, row_bytes, &bar);
    }
  }
  if (threadIdx.x < K) gates[threadIdx.x] = __ldg(gate + static_cast<size_t>(t) * K + threadIdx.x);
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  // every thread waits on the copies; the wait is bounded
  const bool ok = ptx::mbar_wait(&bar, 0u, &abort_flag, timeout_ns);
  if (!__syncthreads_and(ok ? 1 : 0)) {
    if (threadIdx.x == 0) atomicOr(err, DEVERR_TIMEOUT_EPILOGUE);
    // copies still in flight must land before the CTA exits (bounded again)
    ptx::mbar_wait(&bar, 0u, &abort_flag, timeout_ns);
    return;
  }
  combine_staged_rows(reinterpret_cast<const uint4*>(cb_smem), gates, warp_ss, gamma, K, L, eps,
                      z + static_cast<size_t>(t) * ldz);
}

// The same combine with the token's rows staged in rounds of `rpp` (a buffer of rpp rows) and
// two 8-feature vectors per thread: a CTA needs rpp * L * 2 bytes of shared memory and L / 16
// threads, so more tokens are in flight per SM -- four at rpp = 7 and L = 3584 (50 KB and 224
// threads each), against two when all 16 rows of a token are staged at once.  u accumulates in
// the same slot order as combine_bulk_kernel and the norm takes the same tree, so z has that
// kernel's bits (for L <= 4096, where it holds one vector per thread): the choice between the
// two may depend on the batch size without a token's output depending on its batch.
__global__ void __launch_bounds__(COMBINE_MAX_THREADS)
combine_rounds_kernel(const __nv_bfloat16* __restrict__ o, const float* __restrict__ gate,
                      const int32_t* __restrict__ inv, const float* __restrict__ gamma, int T,
                      int K, int L, float eps, __nv_bfloat16* __restrict__ z, int ldz, int rpp,
                      uint32_t* __restrict__ err, unsigned long long timeout_ns) {
  extern __shared__ __align__(128) uint8_t cr_smem[];
  __shared__ float gates[32];
  __shared__ float warp_ss[32];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int t = blockIdx.x;
  const uint32_t row_bytes = static_cast<uint32_t>(L) * 2;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x < K) gates[threadIdx.x] = __ldg(gate + static_cast<size_t>(t) * K + threadIdx.x);
  __syncthreads();
  float u[COMBINE_MAX_VEC][8];
#pragma unroll
  for (int c = 0; c < COMBINE_MAX_VEC; ++c)
#pragma unroll
    for (int i = 0; i < 8; ++i) u[c][i] = 0.0f;
  int round = 0;
  for (int j0 = 0; j0 < K; j0 += rpp, ++round) {
    const int nr = K - j0 < rpp ? K - j0 : rpp;
    if (threadIdx.x == 0) {
      ptx::mbar_arrive_expect_tx(&bar, row_bytes * static_cast<uint32_t>(nr));
      for (int j = 0; j < nr; ++j) {
        const int row = __ldg(inv + static_cast<size_t>(t) * K + j0 + j);
        ptx::bulk_load(cr_smem + static_cast<size_t>(j) * row_bytes,
                       o + static_cast<size_t>(row) * L, row_bytes, &bar);
      }
    }
    const bool ok = ptx::mbar_wait(&bar, static_cast<uint32_t>(round) & 1u, &abort_flag,
                                   timeout_ns);
    if (!__syncthreads_and(ok ? 1 : 0)) {
      if (threadIdx.x == 0) atomicOr(err, DEVERR_TIMEOUT_EPILOGUE);
      // copies still in flight must land before the CTA exits (bounded again)
      ptx::mbar_wait(&bar, static_cast<uint32_t>(round) & 1u, &abort_flag, timeout_ns);
      return;
    }
    combine_accumulate(reinterpret_cast<const uint4*>(cr_smem), gates + j0, nr, L, u);
    __syncthreads();  // every thread is done with the buffer before the next round fills it
  }
  combine_finish_pairs(u, warp_ss, gamma, L, eps, z + static_cast<size_t>(t) * ldz);
}

// ------------------------------------------------------------------------------------
int launch_dispatch(const int32_t* idx, int T, int E, int K, uint32_t* masks, uint32_t* base,
                    int32_t* offsets, int32_t* ct_off, int tokn, int32_t* ct_off2, int tokn2,
                    int32_t* inv, int32_t* src_tok, int32_t* counts_out, uint32_t* err,
                    cudaStream_t stream) {
  if (tokn < 1 || (ct_off2 && tokn2 < 1)) return LMOE_ERR_INVALID_ARG;
  const int nb = static_cast<int>(ceil_div(T, DISPATCH_TOKENS));
  const size_t msmem = static_cast<size_t>(E) * sizeof(uint32_t);
  uint32_t* done = err + 1;  // the word after the error flag
  if (nb > 0) {
    if (launch_pdl(dispatch_mask_kernel, nb, 256, msmem, stream, idx, T, E, K, masks, err, done) !=
        cudaSuccess)
      return LMOE_ERR_CUDA;
  } else if (cudaMemsetAsync(done, 0, sizeof(uint32_t), stream) != cudaSuccess) {
    return LMOE_ERR_CUDA;
  }
  if (launch_pdl(dispatch_scan_kernel, static_cast<unsigned>(ceil_div(E, 32)), SCAN_THREADS, 0,
                 stream, masks, nb, E, base, offsets, ct_off, tokn, ct_off2, tokn2, counts_out,
                 done) !=
      cudaSuccess)
    return LMOE_ERR_CUDA;
  if (nb > 0) {
    const int64_t pairs = static_cast<int64_t>(T) * K;
    if (launch_pdl(dispatch_scatter_kernel, static_cast<unsigned>(ceil_div(pairs, 256)), 256, 0,
                   stream, idx, masks, base, offsets, T, E, K, inv, src_tok) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  return LMOE_OK;
}

int launch_combine(const __nv_bfloat16* o, const float* gate, const int32_t* inv,
                   const float* gamma, int T, int K, int L, float eps, __nv_bfloat16* z,
                   int ldz, uint32_t* err, unsigned long long timeout_ns, cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  const int nvec = L / 8;
  const int threads = static_cast<int>(
      ceil_div(nvec < COMBINE_MAX_THREADS ? nvec : COMBINE_MAX_THREADS, 32) * 32);
  if (nvec > COMBINE_MAX_VEC * threads) return LMOE_ERR_UNSUPPORTED;
  const size_t staged = static_cast<size_t>(K) * L * 2;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  // Rounds pay once tokens queue for the SMs; a batch whose CTAs are all resident at once with
  // the whole-token staging (two per SM) is done in one round trip per token instead of three
  // (decode, T = 64: 6.4 us against 10 us).
  const bool rounds_pay = T > 2 * static_cast<int64_t>(sms) || staged > COMBINE_BULK_MAX;
  // (nvec <= 512: the other kernels hold one vector per thread, whose tree the rounds follow)
  if (COMBINE_ROUND_ROWS > 0 && rounds_pay && K > COMBINE_ROUND_ROWS && nvec >= 64 &&
      nvec <= COMBINE_MAX_THREADS) {
    // rounds of COMBINE_ROUND_ROWS rows, two vectors per thread
    const int th = static_cast<int>(ceil_div(ceil_div(nvec, 2), 32) * 32);
    const size_t sm = static_cast<size_t>(COMBINE_ROUND_ROWS) * L * 2;
    if (cudaFuncSetAttribute(combine_rounds_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sm)) != cudaSuccess)
      return LMOE_ERR_CUDA;
    return launch_pdl(combine_rounds_kernel, T, th, sm, stream, o, gate, inv, gamma, T, K, L,
                      eps, z, ldz, COMBINE_ROUND_ROWS, err, timeout_ns) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  }
  if (staged <= static_cast<size_t>(COMBINE_BULK_MAX)) {
    if (cudaFuncSetAttribute(combine_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(staged)) != cudaSuccess)
      return LMOE_ERR_CUDA;
    return launch_pdl(combine_bulk_kernel, T, threads, staged, stream, o, gate, inv, gamma, T, K,
                      L, eps, z, ldz, err, timeout_ns) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  }
  return launch_pdl(combine_rmsnorm_kernel, T, threads, 0, stream, o, gate, inv, gamma, T, K, L,
                    eps, z, ldz) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

}  // namespace lmoe
