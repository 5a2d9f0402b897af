// routing.cu -- router score, Quantile-Balancing thresholds and top-K selection.
//
// Sources: "The 2.8-Trillion-Parameter Problem: Why Bigger Models Break the Old Playbook"
// (aitrending.vip summary, "Technical Details": a lightweight router selects 16 of 896
// experts per token); the same title, "Part 1 of Inside Kimi K3" (Towards AI article,
// Quantile Balancing passage: thresholds read off the distribution of router scores at
// each step, the score an expert needs to stay within its fair share); "苏神复盘 Kimi K3"
// (daily-ai-frontier, "Merged summary", Stable LatentMoE bullet: solving directly for
// per-expert Top-K thresholds in place of the predecessor's bias updates).
//
// Every decision here is taken in fp32 with explicitly rounded operations (__fmul_rn,
// __fadd_rn, __fmaf_rn, __fdiv_rn), so that no contraction or approximation changes a
// result bit: a CPU evaluation of the same sequence of IEEE operations agrees exactly.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

// Router score s = sigmoid(z) as a fixed sequence of fp32 operations (the pages name no
// score function; the logistic sigmoid is the reading):
//   clamp z to [-88, 88], x = -z
//   Cody-Waite reduction (Cody & Waite 1980): n = rint(x * fl32(1/ln2)),
//     r = fma(-n, ln2_hi, x), r = fma(-n, ln2_lo, r), ln2_hi = 22713/32768 (15 significant
//     bits: n * ln2_hi is exact for |n| <= 127), ln2_lo = fl32(ln2 - ln2_hi)
//   exp(r) by its degree-7 Taylor polynomial, coefficients fl32(1/k!), fma Horner
//   e = (p * 2^(n/2)) * 2^(n - n/2)   (two normal powers of two)
//   s = 1 / (1 + e)
__device__ __forceinline__ float score_sigmoid(float z) {
  z = fminf(fmaxf(z, -88.0f), 88.0f);
  const float x = -z;
  const float nf = rintf(__fmul_rn(x, 0x1.715476p+0f));
  float r = __fmaf_rn(-nf, 0x1.62e4p-1f, x);
  r = __fmaf_rn(-nf, 0x1.7f7d1cp-20f, r);
  float p = 0x1.a01a02p-13f;          // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/3!
  p = __fmaf_rn(p, r, 0.5f);             // 1/2!
  p = __fmaf_rn(p, r, 1.0f);             // 1/1!
  p = __fmaf_rn(p, r, 1.0f);             // 1/0!
  const int n = static_cast<int>(nf);
  const int n1 = n / 2, n2 = n - n1;
  const float s1 = __int_as_float((n1 + 127) << 23);
  const float s2 = __int_as_float((n2 + 127) << 23);
  const float e = __fmul_rn(__fmul_rn(p, s1), s2);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

// Order-preserving map of an fp32 value to uint32 (larger float -> larger key); -0 is
// folded onto +0 first so that the order equals IEEE comparison.
__device__ __forceinline__ uint32_t order_key(float a) {
  a = __fadd_rn(a, 0.0f);
  const uint32_t u = __float_as_uint(a);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------------------------------
// Top-K routing: one warp per token.  The warp writes the token's keys a = fl32(s - tau)
// into shared memory, then K times takes the largest remaining key (ties to the lower
// expert id) with two warp reductions.  Each lane keeps its own best candidate and only
// the lane that lost its candidate rescans its share of the experts.
// ------------------------------------------------------------------------------------
constexpr int ROUTE_WARPS = 4;

__global__ void __launch_bounds__(ROUTE_WARPS * 32)
route_kernel(const float* __restrict__ logits, const float* __restrict__ tau, int T, int E,
             int K, int32_t* __restrict__ idx, float* __restrict__ gate,
             float* __restrict__ scores_out) {
  extern __shared__ uint32_t route_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* keys = route_smem + static_cast<size_t>(warp) * E;
  const int t = blockIdx.x * ROUTE_WARPS + warp;
  if (t >= T) return;
  const float* zrow = logits + static_cast<size_t>(t) * E;

  for (int e = lane; e < E; e += 32) {
    const float s = score_sigmoid(__ldg(zrow + e));
    if (scores_out) scores_out[static_cast<size_t>(t) * E + e] = s;
    const float a = tau ? __fsub_rn(s, __ldg(tau + e)) : s;
    keys[e] = order_key(a);
  }
  __syncwarp();

  // lane-local best among e = lane, lane + 32, ...
  auto lane_best = [&](uint32_t& bk, int& be) {
    bk = 0u;
    be = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const uint32_t k = keys[e];
      if (k > bk) {  // strictly greater keeps the lower e on ties (ascending scan)
        bk = k;
        be = e;
      }
    }
  };
  uint32_t bk;
  int be;
  lane_best(bk, be);
  int my_idx = 0;  // lane j keeps the j-th winner
  for (int j = 0; j < K; ++j) {
    const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
    const int we = static_cast<int>(
        __reduce_min_sync(0xffffffffu, bk == mk ? static_cast<uint32_t>(be) : 0xffffffffu));
    if (lane == j) my_idx = we;
    if (lane == (we & 31)) {
      keys[we] = 0u;  // below every real key
      lane_best(bk, be);
    }
    __syncwarp();
  }
  // gates: s of the winners, fp32 sum in slot order, then one rounded division each
  const float sj = (lane < K) ? score_sigmoid(__ldg(zrow + my_idx)) : 0.0f;
  float sum = 0.0f;
  for (int j = 0; j < K; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, sj, j));
  if (lane < K) {
    idx[static_cast<size_t>(t) * K + lane] = my_idx;
    gate[static_cast<size_t>(t) * K + lane] = __fdiv_rn(sj, sum);
  }
}

// ------------------------------------------------------------------------------------
// Quantile-Balancing thresholds: one CTA per expert column.  The scores of the column
// (non-negative, so their fp32 bit patterns are ordered like their values) are staged in
// shared memory when they fit, then the k-th largest is found by a three-pass radix
// select over bits [31:21], [20:10], [9:0] with shared-memory histograms.
// ------------------------------------------------------------------------------------
constexpr int TH_THREADS = 512;
constexpr int TH_BINS = 2048;
constexpr int TH_SMEM_MAX_T = 32768;

__global__ void __launch_bounds__(TH_THREADS)
thresholds_kernel(const float* __restrict__ logits, int T, int E, int k,
                  float* __restrict__ tau) {
  extern __shared__ uint32_t th_smem[];
  uint32_t* hist = th_smem;                  // [TH_BINS]
  uint32_t* ctl = th_smem + TH_BINS;         // [0] = digit, [1] = new k
  uint32_t* vals = th_smem + TH_BINS + 32;   // [T] when staged
  const int e = blockIdx.x;
  const bool staged = T <= TH_SMEM_MAX_T;
  if (staged) {
    for (int t = threadIdx.x; t < T; t += TH_THREADS)
      vals[t] = __float_as_uint(score_sigmoid(__ldg(logits + static_cast<size_t>(t) * E + e)));
  }
  uint32_t prefix = 0u, mask = 0u;
  int krem = k;
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dm = pass == 2 ? 0x3FFu : 0x7FFu;
    for (int b = threadIdx.x; b < TH_BINS; b += TH_THREADS) hist[b] = 0u;
    __syncthreads();
    for (int t = threadIdx.x; t < T; t += TH_THREADS) {
      const uint32_t key =
          staged ? vals[t]
                 : __float_as_uint(score_sigmoid(__ldg(logits + static_cast<size_t>(t) * E + e)));
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns bins [64 l, 64 l + 64); count of keys in bins above lane l's range
      const int lane = threadIdx.x;
      uint32_t mine = 0u;
      for (int b = 0; b < 64; ++b) mine += hist[lane * 64 + b];
      uint32_t incl = mine;  // inclusive suffix sum over lanes >= lane
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += v;
      }
      const uint32_t above = incl - mine;
      if (above < static_cast<uint32_t>(krem) && static_cast<uint32_t>(krem) <= incl) {
        uint32_t cum = above;
        for (int b = 63; b >= 0; --b) {
          const uint32_t h = hist[lane * 64 + b];
          if (cum + h >= static_cast<uint32_t>(krem)) {
            ctl[0] = static_cast<uint32_t>(lane * 64 + b);
            ctl[1] = static_cast<uint32_t>(krem) - cum;
            break;
          }
          cum += h;
        }
      }
    }
    __syncthreads();
    prefix |= ctl[0] << sh;
    mask |= dm << sh;
    krem = static_cast<int>(ctl[1]);
    __syncthreads();
  }
  if (threadIdx.x == 0) tau[e] = __uint_as_float(prefix);
}

// ------------------------------------------------------------------------------------
// launchers
// ------------------------------------------------------------------------------------
int launch_route(const float* logits, const float* tau, int T, int E, int K, int32_t* idx,
                 float* gate, float* scores_out, cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  const size_t smem = static_cast<size_t>(ROUTE_WARPS) * E * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  const int grid = static_cast<int>(ceil_div(T, ROUTE_WARPS));
  route_kernel<<<grid, ROUTE_WARPS * 32, smem, stream>>>(logits, tau, T, E, K, idx, gate,
                                                         scores_out);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

int launch_thresholds(const float* logits, int T, int E, int k, float* tau,
                      cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  const size_t smem = (TH_BINS + 32 + (T <= TH_SMEM_MAX_T ? T : 0)) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(thresholds_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  thresholds_kernel<<<E, TH_THREADS, smem, stream>>>(logits, T, E, k, tau);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

}  // namespace lmoe
