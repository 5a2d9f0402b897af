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
// __fadd_rn, __fmaf_rn, __fdiv_rn, __frcp_rn), so that no contraction or approximation
// changes a result bit: a CPU evaluation of the same sequence of IEEE operations agrees
// exactly.
#include <cfloat>

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
  return __frcp_rn(__fadd_rn(1.0f, e));  // correctly rounded, so equal to 1.0f / (1 + e)
}

// Order-preserving map of an fp32 value to uint32 (larger float -> larger key); -0 is
// folded onto +0 first so that the order equals IEEE comparison.
__device__ __forceinline__ uint32_t order_key(float a) {
  a = __fadd_rn(a, 0.0f);
  const uint32_t u = __float_as_uint(a);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Score of a routing input: the input itself when it already is a score (SCORES), else the
// score of a logit.
template <bool SCORES>
__device__ __forceinline__ float score_of(float v) {
  return SCORES ? v : score_sigmoid(v);
}

// K rounds of argmax over keys[0..E) in shared memory (consumed), ties to the lower expert
// id: lane j returns the j-th winner (lanes >= K return 0).  Called by a whole warp.
__device__ __forceinline__ int select_rounds(uint32_t* keys, int E, int K, int lane) {
  // best (b1) and runner-up (b2) among e = lane, lane + 32, ...; key 0 = none.  The scan is
  // ascending in e and replaces only on a strictly larger key, so equal keys keep the lower e.
  uint32_t b1k = 0u, b2k = 0u;
  int b1e = 0x7fffffff, b2e = 0x7fffffff;
  auto rescan = [&]() {
    b1k = 0u;
    b2k = 0u;
    b1e = b2e = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const uint32_t k = keys[e];
      if (k > b1k) {
        b2k = b1k;
        b2e = b1e;
        b1k = k;
        b1e = e;
      } else if (k > b2k) {
        b2k = k;
        b2e = e;
      }
    }
  };
  rescan();
  int my_idx = 0;  // lane j keeps the j-th winner
  for (int j = 0; j < K; ++j) {
    const uint32_t mk = __reduce_max_sync(0xffffffffu, b1k);
    const int we = static_cast<int>(
        __reduce_min_sync(0xffffffffu, b1k == mk ? static_cast<uint32_t>(b1e) : 0xffffffffu));
    if (lane == j) my_idx = we;
    if (lane == (we & 31)) {
      keys[we] = 0u;  // below every real key
      if (b2k != 0u) {
        b1k = b2k;
        b1e = b2e;
        b2k = 0u;  // runner-up unknown now: rescan if this lane wins again
        b2e = 0x7fffffff;
      } else {
        rescan();
      }
    }
    __syncwarp();
  }
  return my_idx;
}

// ------------------------------------------------------------------------------------
// Top-K routing: one warp per token.  The warp writes the token's keys a = fl32(s - tau)
// into shared memory, then K times takes the largest remaining key (ties to the lower
// expert id) with two warp reductions.  Each lane keeps its best and second-best candidate,
// so a lane whose best is taken promotes its runner-up and only rescans its share of the
// experts when it loses a second time.
// ------------------------------------------------------------------------------------
constexpr int ROUTE_WARPS = 4;

template <bool SCORES>
__global__ void __launch_bounds__(ROUTE_WARPS * 32)
route_kernel(const float* __restrict__ logits, const float* __restrict__ tau, int T, int E,
             int K, int32_t* __restrict__ idx, float* __restrict__ gate,
             float* __restrict__ scores_out) {
  extern __shared__ uint32_t route_smem[];
  pdl_wait();
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* keys = route_smem + static_cast<size_t>(warp) * E;
  const int t = blockIdx.x * ROUTE_WARPS + warp;
  if (t >= T) return;
  const float* zrow = logits + static_cast<size_t>(t) * E;

  // eight independent logit loads in flight per lane before their keys are computed
  constexpr int B = 8;
  for (int e0 = lane; e0 < E; e0 += B * 32) {
    float zv[B], tv[B];
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int e = e0 + i * 32;
      zv[i] = e < E ? __ldg(zrow + e) : 0.0f;
      tv[i] = (tau && e < E) ? __ldg(tau + e) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int e = e0 + i * 32;
      if (e < E) {
        const float s = score_of<SCORES>(zv[i]);
        if (scores_out) scores_out[static_cast<size_t>(t) * E + e] = s;
        const float a = tau ? __fsub_rn(s, tv[i]) : s;
        keys[e] = order_key(a);
      }
    }
  }
  __syncwarp();

  const int my_idx = select_rounds(keys, E, K, lane);
  // gates: s of the winners, fp32 sum in slot order, then one rounded division each
  const float sj = (lane < K) ? score_of<SCORES>(__ldg(zrow + my_idx)) : 0.0f;
  float sum = 0.0f;
  for (int j = 0; j < K; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, sj, j));
  if (lane < K) {
    idx[static_cast<size_t>(t) * K + lane] = my_idx;
    gate[static_cast<size_t>(t) * K + lane] = __fdiv_rn(sj, sum);
  }
}

// ------------------------------------------------------------------------------------
// Top-K routing, register form (E a multiple of 4 and at most 4 * 32 * RF_NQ, rows 16-byte
// aligned): one warp per token, lane l holding the keys of experts 4(l + 32q) + c in
// registers, the CTA's thresholds in shared memory.  The K-th largest of the lanes' maxima
// is a lower bound B on the token's K-th largest key (K lanes each hold a key >= B).  The
// winners, in order (larger key first, then the lower expert id), are then found among few
// keys:
//   - at most RF_CAND keys >= B: each is ranked against the others;
//   - else, fewer than K keys > B (many keys equal to B, as when scores saturate at 1 and
//     so do the thresholds): the keys > B ranked as above, then the experts whose key is B
//     in ascending id;
//   - else K rounds of argmax over all E keys in shared memory.
// Each gives the same experts in the same order as K rounds of argmax.
// ------------------------------------------------------------------------------------
constexpr int RF_WARPS = 8;
constexpr int RF_NQ = 8;      // float4 of logits per lane: E <= 1024
constexpr int RF_CAND = 64;   // candidates ranked in place
constexpr int RF_WARP_WORDS = 2 * RF_CAND + 32;  // + E words for the last form

template <bool SCORES>
__global__ void __launch_bounds__(RF_WARPS * 32, 3)
route_reg_kernel(const float* __restrict__ logits, const float* __restrict__ tau, int T, int E,
                 int K, int32_t* __restrict__ idx, float* __restrict__ gate,
                 float* __restrict__ scores_out) {
  extern __shared__ uint32_t rf_smem[];
  pdl_wait();
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = E >> 2;
  float4* tau_s = reinterpret_cast<float4*>(rf_smem);  // [nq] (zeros without thresholds)
  for (int j = threadIdx.x; j < nq; j += RF_WARPS * 32)
    tau_s[j] = tau ? __ldg(reinterpret_cast<const float4*>(tau) + j)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  uint32_t* ckey = rf_smem + E + static_cast<size_t>(warp) * (RF_WARP_WORDS + E);
  int32_t* ce = reinterpret_cast<int32_t*>(ckey + RF_CAND);
  int32_t* sel = ce + RF_CAND;                                  // [32] winners by slot
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel + 32);       // [E] last form
  const int t = blockIdx.x * RF_WARPS + warp;
  if (t >= T) return;
  const float* zrow = logits + static_cast<size_t>(t) * E;

  float4 zv[RF_NQ];
#pragma unroll
  for (int q = 0; q < RF_NQ; ++q) {
    const int j = lane + 32 * q;
    zv[q] = j < nq ? __ldg(reinterpret_cast<const float4*>(zrow) + j)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // keys; 0 marks no expert (every finite a has a key >= 1)
  uint32_t key[4 * RF_NQ];
#pragma unroll
  for (int i = 0; i < 4 * RF_NQ; ++i) key[i] = 0u;
  uint32_t mk = 0u;
#pragma unroll
  for (int q = 0; q < RF_NQ; ++q) {
    if (32 * q >= nq) break;  // warp-uniform: no lane holds experts past this row
    const int j = lane + 32 * q;
    if (j < nq) {
      const float4 tq = tau_s[j];
      const float zz[4] = {zv[q].x, zv[q].y, zv[q].z, zv[q].w};
      const float tt[4] = {tq.x, tq.y, tq.z, tq.w};
      float ss[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        ss[c] = score_of<SCORES>(zz[c]);
        key[4 * q + c] = order_key(tau ? __fsub_rn(ss[c], tt[c]) : ss[c]);
        mk = key[4 * q + c] > mk ? key[4 * q + c] : mk;
      }
      if (scores_out)
        reinterpret_cast<float4*>(scores_out + static_cast<size_t>(t) * E)[j] =
            make_float4(ss[0], ss[1], ss[2], ss[3]);
    }
  }
  // B = the K-th largest lane maximum: bitonic sort of the 32 maxima (ascending), lane 32 - K
  uint32_t v = mk;
#pragma unroll
  for (int w = 2; w <= 32; w <<= 1) {
#pragma unroll
    for (int j = w >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool up = (lane & w) == 0, lower = (lane & j) == 0;
      v = (lower == up) ? (o < v ? o : v) : (o > v ? o : v);
    }
  }
  const uint32_t bound = __shfl_sync(0xffffffffu, v, 32 - K);
  int c_ge = 0, c_gt = 0;
#pragma unroll
  for (int i = 0; i < 4 * RF_NQ; ++i) {
    c_ge += (key[i] != 0u && key[i] >= bound) ? 1 : 0;
    c_gt += key[i] > bound ? 1 : 0;
  }
  const int n_ge = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(c_ge));
  const int n_gt = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(c_gt));
  // rank the keys >= B (strict = false) or > B (strict = true) against each other
  auto rank_keys = [&](bool strict, int cnt, int n) {
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    int p = incl - cnt;
#pragma unroll
    for (int i = 0; i < 4 * RF_NQ; ++i) {
      if (key[i] != 0u && (strict ? key[i] > bound : key[i] >= bound)) {
        ckey[p] = key[i];
        ce[p] = 4 * (lane + 32 * (i >> 2)) + (i & 3);
        ++p;
      }
    }
    __syncwarp();
    for (int m0 = lane; m0 < n; m0 += 32) {
      const uint32_t km = ckey[m0];
      const int em = ce[m0];
      int rank = 0;
      for (int m = 0; m < n; ++m) {
        const uint32_t k2 = ckey[m];
        rank += (k2 > km || (k2 == km && ce[m] < em)) ? 1 : 0;
      }
      if (rank < K) sel[rank] = em;
    }
  };
  int my_idx = 0;
  if (n_ge <= RF_CAND) {
    rank_keys(false, c_ge, n_ge);
    __syncwarp();
    if (lane < K) my_idx = sel[lane];
  } else if (n_gt < K) {
    rank_keys(true, c_gt, n_gt);
    // slots n_gt .. K-1: the experts whose key is B, in ascending id (row q, then lane, then c)
    int filled = n_gt;
#pragma unroll
    for (int q = 0; q < RF_NQ; ++q) {
      if (32 * q >= nq || filled >= K) break;  // warp-uniform
      uint32_t f = 0u;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        f |= (key[4 * q + c] != 0u && key[4 * q + c] == bound) ? (1u << c) : 0u;
      const int cnt = __popc(f);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      int slot = filled + incl - cnt;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (f & (1u << c)) {
          if (slot < K) sel[slot] = 4 * (lane + 32 * q) + c;
          ++slot;
        }
      }
      filled += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    if (lane < K) my_idx = sel[lane];
  } else {
#pragma unroll
    for (int i = 0; i < 4 * RF_NQ; ++i) {
      const int j = lane + 32 * (i >> 2);
      if (j < nq) keys[4 * j + (i & 3)] = key[i];
    }
    __syncwarp();
    my_idx = select_rounds(keys, E, K, lane);
  }
  // gates: s of the winners, fp32 sum in slot order, then one rounded division each
  const float sj = (lane < K) ? score_of<SCORES>(__ldg(zrow + my_idx)) : 0.0f;
  float sum = 0.0f;
  for (int j = 0; j < K; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, sj, j));
  if (lane < K) {
    idx[static_cast<size_t>(t) * K + lane] = my_idx;
    gate[static_cast<size_t>(t) * K + lane] = __fdiv_rn(sj, sum);
  }
}

// ------------------------------------------------------------------------------------
// Quantile-Balancing thresholds: one CTA per expert.  The scores of the expert's column
// (non-negative, so their fp32 bit patterns order like their values, and below 2^30) are
// staged in shared memory when they fit; the k-th largest is then found by a radix select
// over bits [29:18], [17:9], [8:0].  After a pass whose selected bin holds at most
// TH_CAND keys, those keys are compacted and the remaining passes read only them (for the
// fair-share rank that is ~2 % of the column).  Histograms use shared-memory atomics.
// ------------------------------------------------------------------------------------
constexpr int TH_THREADS = 256;
constexpr int TH_BINS = 4096;
constexpr int TH_CAND = 4096;
constexpr int TH_SMEM_MAX_T = 32768;
static_assert(512 % TH_THREADS == 0 && TH_THREADS / 32 <= 8, "bin ranges and warp sums");

struct KthResult {
  uint32_t key;  // score bits of the k-th largest score of the column
  int above;     // number of scores strictly greater than it (< k)
};

// k-th largest score (1 <= k <= T) of column `col` (T logits, stride stride_t).  Called by
// all TH_THREADS threads of the CTA; `th_smem` is the layout launch_thresholds sizes.  When
// the column is staged, vals[0..T) keeps the score bits on return.
template <bool SCORES>
__device__ __forceinline__ KthResult select_kth_score(const float* __restrict__ col, int T,
                                                     int64_t stride_t, int k,
                                                     uint32_t* th_smem, bool staged) {
  uint32_t* hist = th_smem;                       // [TH_BINS]
  uint32_t* ctl = th_smem + TH_BINS;              // [0] digit, [1] new k, [2] in bin,
                                                  // [3] count, [8..16) warp sums
  uint32_t* cand = th_smem + TH_BINS + 32;        // [TH_CAND]
  uint32_t* vals = cand + TH_CAND;                // [T] when staged
  const int lane = threadIdx.x & 31;
  if (staged) {
    // eight independent loads in flight per thread before their scores are computed
    constexpr int B = 8;
    for (int t0 = threadIdx.x; t0 < T; t0 += B * TH_THREADS) {
      float zv[B];
#pragma unroll
      for (int i = 0; i < B; ++i) {
        const int t = t0 + i * TH_THREADS;
        zv[i] = t < T ? __ldg(col + t * stride_t) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < B; ++i) {
        const int t = t0 + i * TH_THREADS;
        if (t < T) vals[t] = __float_as_uint(score_of<SCORES>(zv[i]));
      }
    }
  }
  // source of the keys: the full column (staged or re-read), or the compacted candidates
  bool from_cand = false;
  int n = T;
  auto key_at = [&](int i) -> uint32_t {
    if (from_cand) return cand[i];
    return staged ? vals[i] : __float_as_uint(score_of<SCORES>(__ldg(col + i * stride_t)));
  };
  uint32_t prefix = 0u, mask = 0u;
  int krem = k;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 18 : (pass == 1 ? 9 : 0);
    const uint32_t dm = pass == 0 ? 0xFFFu : 0x1FFu;
    const int nbins = static_cast<int>(dm) + 1;
    for (int b = threadIdx.x; b < nbins; b += TH_THREADS) hist[b] = 0u;
    __syncthreads();
    const int n_round = (n + 31) & ~31;  // whole warps iterate together
    for (int i = threadIdx.x; i < n_round; i += TH_THREADS) {
      uint32_t key = 0u;
      bool in = false;
      if (i < n) {
        key = key_at(i);
        in = (key & mask) == prefix;
      }
      if (in) atomicAdd(&hist[(key >> sh) & dm], 1u);
    }
    __syncthreads();
    {
      // thread i owns bins [per i, per i + per); a block-wide suffix sum gives the count
      // above its range, and the one thread whose range holds the krem-th key finds its bin
      const int per = nbins / TH_THREADS;
      const int warp = threadIdx.x >> 5;
      const int b0 = threadIdx.x * per;
      uint32_t mine = 0u;  // neighbouring lanes start at different banks
      for (int b = 0; b < per; ++b) mine += hist[b0 + ((b + lane) & (per - 1))];
      uint32_t incl = mine;  // inclusive suffix sum over the lanes >= lane of this warp
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += v;
      }
      if (lane == 0) ctl[8 + warp] = incl;  // warp total
      __syncthreads();
      uint32_t above_w = 0u;  // keys in the warps above this one
      for (int w = warp + 1; w < TH_THREADS / 32; ++w) above_w += ctl[8 + w];
      const uint32_t above = above_w + incl - mine;
      if (above < static_cast<uint32_t>(krem) && static_cast<uint32_t>(krem) <= above + mine) {
        uint32_t cum = above;
        for (int b = per - 1; b >= 0; --b) {
          const uint32_t h = hist[b0 + b];
          if (cum + h >= static_cast<uint32_t>(krem)) {
            ctl[0] = static_cast<uint32_t>(b0 + b);
            ctl[1] = static_cast<uint32_t>(krem) - cum;
            ctl[2] = h;
            break;
          }
          cum += h;
        }
      }
    }
    __syncthreads();
    const uint32_t digit = ctl[0];
    const uint32_t in_bin = ctl[2];
    prefix |= digit << sh;
    mask |= dm << sh;
    krem = static_cast<int>(ctl[1]);
    if (pass < 2 && !from_cand && in_bin <= static_cast<uint32_t>(TH_CAND)) {
      // compact the keys of the selected bin (warp-aggregated appends)
      if (threadIdx.x == 0) ctl[3] = 0u;
      __syncthreads();
      for (int i = threadIdx.x; i < n_round; i += TH_THREADS) {
        uint32_t key = 0u;
        bool in = false;
        if (i < n) {
          key = key_at(i);
          in = (key & mask) == prefix;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, in);
        uint32_t base = 0u;
        if (lane == 0 && bal) base = atomicAdd(&ctl[3], static_cast<uint32_t>(__popc(bal)));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (in) cand[base + __popc(bal & ((1u << lane) - 1u))] = key;
      }
      __syncthreads();
      from_cand = true;
      n = static_cast<int>(ctl[3]);
    }
    __syncthreads();
  }
  // after the last pass the selected bin is one key value; krem of its copies complete k
  KthResult r;
  r.key = prefix;
  r.above = k - krem;
  return r;
}

template <bool SCORES>
__global__ void __launch_bounds__(TH_THREADS)
thresholds_kernel(const float* __restrict__ z, int T, int64_t stride_t, int64_t stride_e,
                  int k, float* __restrict__ tau) {
  extern __shared__ uint32_t th_smem[];
  pdl_wait();
  pdl_launch_dependents();

  const int e = blockIdx.x;
  const KthResult r = select_kth_score<SCORES>(z + static_cast<int64_t>(e) * stride_e, T,
                                               stride_t, k, th_smem, T <= TH_SMEM_MAX_T);
  if (threadIdx.x == 0) tau[e] = __uint_as_float(r.key);
}

// Quantile-Balancing thresholds for columns of at most TH_THREADS * TH_KPT tokens and
// k <= TH_THREADS (SCORES: the columns hold router scores, not logits): one CTA per expert,
// thread i holding the scores of tokens i, i + 256, ... in registers.  The k-th largest of
// the threads' maxima is a lower bound B on the column's k-th largest score (k threads each
// hold a score >= B).  If fewer than k scores exceed B, the k-th largest is B itself (as
// when the top of a column saturates at 1); otherwise it is the k-th largest of the scores
// > B -- about 2.5 % of the column when k is the fair-share rank.  Both selections are
// bit-by-bit searches for the largest v with #{keys >= v} >= k, counted with
// __syncthreads_count.  More than TH_BCAND scores > B falls back to the radix select over
// the whole column.
constexpr int TH_KPT = 32;
constexpr int TH_BCAND = 1024;
static_assert(TH_BCAND <= TH_CAND && TH_BCAND % TH_THREADS == 0, "candidate buffer");

template <bool SCORES>
__global__ void __launch_bounds__(TH_THREADS)
thresholds_bound_kernel(const float* __restrict__ z, int T, int64_t stride_t, int64_t stride_e,
                        int k, float* __restrict__ tau) {
  extern __shared__ uint32_t th_smem[];
  pdl_wait();
  pdl_launch_dependents();

  uint32_t* ctl = th_smem + TH_BINS;         // [3]: count of scores > B
  uint32_t* cand = th_smem + TH_BINS + 32;   // [TH_BCAND]
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const float* col = z + static_cast<int64_t>(e) * stride_e;
  if (threadIdx.x == 0) ctl[3] = 0u;

  // score bits (non-negative, below 2^30); past T a key is 0, which no search value reaches.
  // All the thread's logits are loaded first (one round trip), then scored in place.
  uint32_t key[TH_KPT];
#pragma unroll
  for (int i = 0; i < TH_KPT; ++i) {
    const int t = static_cast<int>(threadIdx.x) + i * TH_THREADS;
    key[i] = t < T ? __float_as_uint(__ldg(col + t * stride_t)) : 0u;
  }
  uint32_t mx = 0u;
#pragma unroll
  for (int i = 0; i < TH_KPT; ++i) {
    const int t = static_cast<int>(threadIdx.x) + i * TH_THREADS;
    key[i] = t < T ? __float_as_uint(score_of<SCORES>(__uint_as_float(key[i]))) : 0u;
    mx = key[i] > mx ? key[i] : mx;
  }
  // B = the k-th largest of the threads' maxima
  uint32_t bound = 0u;
#pragma unroll 1
  for (int b = 29; b >= 0; --b) {
    const uint32_t v = bound | (1u << b);
    if (__syncthreads_count(mx >= v) >= k) bound = v;
  }
  // scores > B: a warp scan of the threads' counts, one shared atomic per warp
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < TH_KPT; ++i) cnt += key[i] > bound ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  uint32_t base = 0u;
  if (lane == 31) base = atomicAdd(&ctl[3], static_cast<uint32_t>(incl));
  base = __shfl_sync(0xffffffffu, base, 31) + static_cast<uint32_t>(incl - cnt);
  __syncthreads();
  const uint32_t n = ctl[3];
  uint32_t result = bound;
  if (n >= static_cast<uint32_t>(k) && n <= static_cast<uint32_t>(TH_BCAND)) {
    uint32_t p = base;
#pragma unroll
    for (int i = 0; i < TH_KPT; ++i)
      if (key[i] > bound) cand[p++] = key[i];
    __syncthreads();
    constexpr int SLOTS = TH_BCAND / TH_THREADS;
    const int used = (static_cast<int>(n) + TH_THREADS - 1) / TH_THREADS;  // block-uniform
    uint32_t cv[SLOTS];
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      const uint32_t q = threadIdx.x + j * TH_THREADS;
      cv[j] = q < n ? cand[q] : 0u;
    }
    result = 0u;
#pragma unroll 1
    for (int b = 29; b >= 0; --b) {
      const uint32_t v = result | (1u << b);
      int c = 0;
#pragma unroll
      for (int j = 0; j < SLOTS; ++j)
        if (j < used) c += __syncthreads_count(cv[j] >= v);
      if (c >= k) result = v;
    }
  } else if (n > static_cast<uint32_t>(TH_BCAND)) {
    result = select_kth_score<SCORES>(col, T, stride_t, k, th_smem, false).key;
  }
  if (threadIdx.x == 0) tau[e] = __uint_as_float(result);
}

// Quantile-Balancing thresholds for columns of at most THR_THREADS * THR_KPT = 32768 tokens and
// any rank k (the bound form above needs k <= 256 and T <= 8192): one CTA of 1024 threads per
// expert, thread i holding the scores of tokens i, i + 1024, ... in registers.  A bit-by-bit
// search finds the largest v with #{scores >= v} >= k -- the k-th largest score -- each count
// a block-wide sum: the threads' own counts, a warp reduction, then one warp over the 32 warp
// sums (double-buffered, two barriers per bit).  Score bits are non-negative and below 2^30;
// past T a key is 0, which no search value reaches.
constexpr int THR_THREADS = 1024;
constexpr int THR_KPT = 32;

template <bool SCORES>
__global__ void __launch_bounds__(THR_THREADS, 1)
thresholds_regs_kernel(const float* __restrict__ z, int T, int64_t stride_t, int64_t stride_e,
                       int k, float* __restrict__ tau) {
  __shared__ uint32_t wsum[2][THR_THREADS / 32];
  __shared__ uint32_t total[2];
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* col = z + static_cast<int64_t>(e) * stride_e;
  uint32_t key[THR_KPT];
#pragma unroll
  for (int i = 0; i < THR_KPT; ++i) {  // every load in flight before any score is computed
    const int t = static_cast<int>(threadIdx.x) + i * THR_THREADS;
    key[i] = t < T ? __float_as_uint(__ldg(col + t * stride_t)) : 0u;
  }
#pragma unroll
  for (int i = 0; i < THR_KPT; ++i) {
    const int t = static_cast<int>(threadIdx.x) + i * THR_THREADS;
    key[i] = t < T ? __float_as_uint(score_of<SCORES>(__uint_as_float(key[i]))) : 0u;
  }
  uint32_t result = 0u;
#pragma unroll 1
  for (int b = 29; b >= 0; --b) {
    const uint32_t v = result | (1u << b);
    uint32_t c = 0u;
#pragma unroll
    for (int i = 0; i < THR_KPT; ++i) c += key[i] >= v ? 1u : 0u;
    c = __reduce_add_sync(0xffffffffu, c);
    const int par = b & 1;
    if (lane == 0) wsum[par][warp] = c;
    __syncthreads();
    if (warp == 0) {
      const uint32_t sum = __reduce_add_sync(0xffffffffu, wsum[par][lane]);
      if (lane == 0) total[par] = sum;
    }
    __syncthreads();
    if (total[par] >= static_cast<uint32_t>(k)) result = v;
  }
  if (threadIdx.x == 0) tau[e] = __uint_as_float(result);
}

// The bound-and-select form for columns of up to THR_THREADS * THR_KPT = 32768 tokens and
// k <= THR_THREADS: one CTA of 1024 threads per expert, thread i holding the scores of tokens
// i, i + 1024, ... in registers.  B, the k-th largest of the threads' maxima, bounds the k-th
// largest score from below; at the fair-share rank ~2.6 % of a column's scores exceed it (the
// skewed workload: ~850 of 32768 for k = 585), so the second bit search runs over at most
// THW_BCAND candidates, a few per thread, with one barrier per bit instead of a block-wide
// reduction of 32 keys per thread.  More than THW_BCAND scores > B: the bit search over the
// registers, as in thresholds_regs_kernel.
constexpr int THW_BCAND = 4096;
static_assert(THW_BCAND % THR_THREADS == 0, "candidate slots per thread");

template <bool SCORES>
__global__ void __launch_bounds__(THR_THREADS, 1)
thresholds_wide_kernel(const float* __restrict__ z, int T, int64_t stride_t, int64_t stride_e,
                       int k, float* __restrict__ tau) {
  __shared__ uint32_t cand[THW_BCAND];
  __shared__ uint32_t wsum[2][THR_THREADS / 32];
  __shared__ uint32_t total[2];
  __shared__ uint32_t ncand;
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* col = z + static_cast<int64_t>(e) * stride_e;
  if (threadIdx.x == 0) ncand = 0u;
  uint32_t key[THR_KPT];
#pragma unroll
  for (int i = 0; i < THR_KPT; ++i) {  // every load in flight before any score is computed
    const int t = static_cast<int>(threadIdx.x) + i * THR_THREADS;
    key[i] = t < T ? __float_as_uint(__ldg(col + t * stride_t)) : 0u;
  }
  uint32_t mx = 0u;
#pragma unroll
  for (int i = 0; i < THR_KPT; ++i) {
    const int t = static_cast<int>(threadIdx.x) + i * THR_THREADS;
    key[i] = t < T ? __float_as_uint(score_of<SCORES>(__uint_as_float(key[i]))) : 0u;
    mx = key[i] > mx ? key[i] : mx;
  }
  // B = the k-th largest of the threads' maxima
  uint32_t bound = 0u;
#pragma unroll 1
  for (int b = 29; b >= 0; --b) {
    const uint32_t v = bound | (1u << b);
    if (__syncthreads_count(mx >= v) >= k) bound = v;
  }
  // scores > B: a warp scan of the threads' counts, one shared atomic per warp
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < THR_KPT; ++i) cnt += key[i] > bound ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  uint32_t base = 0u;
  if (lane == 31) base = atomicAdd(&ncand, static_cast<uint32_t>(incl));
  base = __shfl_sync(0xffffffffu, base, 31) + static_cast<uint32_t>(incl - cnt);
  __syncthreads();
  const uint32_t n = ncand;  // block-uniform
  uint32_t result = bound;
  if (n >= static_cast<uint32_t>(k) && n <= static_cast<uint32_t>(THW_BCAND)) {
    uint32_t p = base;
#pragma unroll
    for (int i = 0; i < THR_KPT; ++i)
      if (key[i] > bound) cand[p++] = key[i];
    __syncthreads();
    constexpr int SLOTS = THW_BCAND / THR_THREADS;
    const int used = (static_cast<int>(n) + THR_THREADS - 1) / THR_THREADS;  // block-uniform
    uint32_t cv[SLOTS];
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      const uint32_t q = threadIdx.x + j * THR_THREADS;
      cv[j] = q < n ? cand[q] : 0u;
    }
    result = 0u;
#pragma unroll 1
    for (int b = 29; b >= 0; --b) {
      const uint32_t v = result | (1u << b);
      int c = 0;
#pragma unroll
      for (int j = 0; j < SLOTS; ++j)
        if (j < used) c += __syncthreads_count(cv[j] >= v);
      if (c >= k) result = v;
    }
  } else if (n > static_cast<uint32_t>(THW_BCAND)) {
    // the whole column's bit search over the registers (block-uniform branch)
    result = 0u;
#pragma unroll 1
    for (int b = 29; b >= 0; --b) {
      const uint32_t v = result | (1u << b);
      uint32_t c = 0u;
#pragma unroll
      for (int i = 0; i < THR_KPT; ++i) c += key[i] >= v ? 1u : 0u;
      c = __reduce_add_sync(0xffffffffu, c);
      const int par = b & 1;
      if (lane == 0) wsum[par][warp] = c;
      __syncthreads();
      if (warp == 0) {
        const uint32_t sum = __reduce_add_sync(0xffffffffu, wsum[par][lane]);
        if (lane == 0) total[par] = sum;
      }
      __syncthreads();
      if (total[par] >= static_cast<uint32_t>(k)) result = v;
    }
  }
  if (threadIdx.x == 0) tau[e] = __uint_as_float(result);
}

// Threshold candidates of one batch: column e of cand ([k, E], row stride ldc) receives the
// logits of the min(k, T) tokens with the largest scores of expert e -- first those whose
// score is above the min(k, T)-th largest, then tokens whose score equals it, both in token
// order -- and rows T..k-1 (when T < k) receive -FLT_MAX, whose score is the lowest any
// logit has.  The k-th largest score of the union of several batches' candidates is the
// k-th largest score of the union of the batches.
__global__ void __launch_bounds__(TH_THREADS)
candidates_kernel(const float* __restrict__ z, int T, int64_t stride_t, int64_t stride_e,
                  int k, float* __restrict__ cand, int64_t ldc) {
  extern __shared__ uint32_t th_smem[];
  pdl_wait();
  pdl_launch_dependents();

  __shared__ uint32_t wsum[2][TH_THREADS / 32];
  __shared__ uint32_t run[2];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* col = z + static_cast<int64_t>(e) * stride_e;
  const int kk = k < T ? k : T;
  if (kk > 0) {
  const bool staged = T <= TH_SMEM_MAX_T;
  const KthResult r = select_kth_score<false>(col, T, stride_t, kk, th_smem, staged);
  const uint32_t* vals = th_smem + TH_BINS + 32 + TH_CAND;
  const int take_eq = kk - r.above;  // copies of the k-th score to emit
  if (threadIdx.x == 0) run[0] = run[1] = 0u;
  __syncthreads();
  // ordered compaction, TH_THREADS tokens per round: warp ballots, then a scan of the
  // warps' counts; run[] carries the counts of earlier rounds
  for (int t0 = 0; t0 < T; t0 += TH_THREADS) {
    const int t = t0 + threadIdx.x;
    bool gt = false, eq = false;
    if (t < T) {
      const uint32_t key =
          staged ? vals[t] : __float_as_uint(score_sigmoid(__ldg(col + t * stride_t)));
      gt = key > r.key;
      eq = key == r.key;
    }
    const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) {
      wsum[0][warp] = __popc(bg);
      wsum[1][warp] = __popc(be);
    }
    __syncthreads();
    uint32_t pg = run[0], pe = run[1];
    for (int w = 0; w < warp; ++w) {
      pg += wsum[0][w];
      pe += wsum[1][w];
    }
    const uint32_t below = (1u << lane) - 1u;
    pg += __popc(bg & below);
    pe += __popc(be & below);
    if (gt) cand[static_cast<int64_t>(pg) * ldc + e] = __ldg(col + t * stride_t);
    if (eq && pe < static_cast<uint32_t>(take_eq))
      cand[static_cast<int64_t>(r.above + pe) * ldc + e] = __ldg(col + t * stride_t);
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t sg = 0u, se = 0u;
      for (int w = 0; w < TH_THREADS / 32; ++w) {
        sg += wsum[0][w];
        se += wsum[1][w];
      }
      run[0] += sg;
      run[1] += se;
    }
    __syncthreads();
  }
  }
  for (int j = kk + threadIdx.x; j < k; j += TH_THREADS)
    cand[static_cast<int64_t>(j) * ldc + e] = -FLT_MAX;
}

// out[E, T] = in[T, E]^T through 32 x 32 shared-memory tiles.
__global__ void __launch_bounds__(256)
transpose_f32_kernel(const float* __restrict__ in, int T, int E, float* __restrict__ out) {
  __shared__ float tile[32][33];
  pdl_wait();
  pdl_launch_dependents();

  const int e0 = blockIdx.x * 32, t0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int i = ty; i < 32; i += 8) {
    const int t = t0 + i, e = e0 + tx;
    if (t < T && e < E) tile[i][tx] = __ldg(in + static_cast<size_t>(t) * E + e);
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + i, t = t0 + tx;
    if (t < T && e < E) out[static_cast<size_t>(e) * T + t] = tile[tx][i];
  }
}

// Router scores, each computed once: s[t, e] = score(z[t, e]) row-major for the top-K
// selection and, when s_t is given, s_t[e, t] expert-major for the thresholds, through
// 32 x 32 shared-memory tiles (each thread's four logits are loaded before any is scored).
__global__ void __launch_bounds__(256)
scores_kernel(const float* __restrict__ z, int T, int E, float* __restrict__ s,
              float* __restrict__ s_t) {
  __shared__ float tile[32][33];
  pdl_wait();
  pdl_launch_dependents();

  const int e0 = blockIdx.x * 32, t0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const int e = e0 + tx;
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty + 8 * i;
    v[i] = (t < T && e < E) ? __ldg(z + static_cast<size_t>(t) * E + e) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty + 8 * i;
    v[i] = score_sigmoid(v[i]);
    if (t < T && e < E) s[static_cast<size_t>(t) * E + e] = v[i];
    tile[ty + 8 * i][tx] = v[i];
  }
  if (!s_t) return;  // grid-uniform
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int er = e0 + ty + 8 * i, t = t0 + tx;
    if (t < T && er < E) s_t[static_cast<size_t>(er) * T + t] = tile[tx][ty + 8 * i];
  }
}

// ------------------------------------------------------------------------------------
// launchers
// ------------------------------------------------------------------------------------
int launch_route(const float* logits, const float* tau, int T, int E, int K, int32_t* idx,
                 float* gate, float* scores_out, bool scores, cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (E % 4 == 0 && E <= 4 * 32 * RF_NQ && a16(logits) && (!tau || a16(tau)) &&
      (!scores_out || a16(scores_out))) {
    const size_t smem =
        (E + static_cast<size_t>(RF_WARPS) * (RF_WARP_WORDS + E)) * sizeof(uint32_t);
    const int grid = static_cast<int>(ceil_div(T, RF_WARPS));
    auto kern = scores ? route_reg_kernel<true> : route_reg_kernel<false>;
    return launch_pdl(kern, grid, RF_WARPS * 32, smem, stream, logits, tau, T, E, K, idx, gate,
                      scores_out) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  }
  const size_t smem = static_cast<size_t>(ROUTE_WARPS) * E * sizeof(uint32_t);
  auto kern = scores ? route_kernel<true> : route_kernel<false>;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  const int grid = static_cast<int>(ceil_div(T, ROUTE_WARPS));
  return launch_pdl(kern, grid, ROUTE_WARPS * 32, smem, stream, logits, tau, T, E, K, idx, gate,
                    scores_out) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_thresholds(const float* z, int T, int E, int64_t stride_t, int64_t stride_e, int k,
                      float* tau, bool scores, cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  if (T <= TH_THREADS * TH_KPT && k <= TH_THREADS) {
    // bound-and-select form; its fallback uses the histogram and candidate buffers
    const size_t smem = (TH_BINS + 32 + TH_CAND) * sizeof(uint32_t);
    auto kern = scores ? thresholds_bound_kernel<true> : thresholds_bound_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LMOE_ERR_CUDA;
    return launch_pdl(kern, E, TH_THREADS, smem, stream, z, T, stride_t, stride_e, k, tau) ==
                   cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  }
  if (T <= THR_THREADS * THR_KPT && k <= THR_THREADS) {
    // bound-and-select with 1024 threads: up to 32768 tokens, k <= 1024
    auto kern = scores ? thresholds_wide_kernel<true> : thresholds_wide_kernel<false>;
    return launch_pdl(kern, E, THR_THREADS, 0, stream, z, T, stride_t, stride_e, k, tau) ==
                   cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  }
  if (T <= THR_THREADS * THR_KPT) {
    // register-resident bit search: any k, up to 32768 tokens
    auto kern = scores ? thresholds_regs_kernel<true> : thresholds_regs_kernel<false>;
    return launch_pdl(kern, E, THR_THREADS, 0, stream, z, T, stride_t, stride_e, k, tau) ==
                   cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  }
  const size_t smem =
      (TH_BINS + 32 + TH_CAND + (T <= TH_SMEM_MAX_T ? T : 0)) * sizeof(uint32_t);
  auto kern = scores ? thresholds_kernel<true> : thresholds_kernel<false>;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  return launch_pdl(kern, E, TH_THREADS, smem, stream, z, T, stride_t, stride_e, k, tau) ==
                 cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_scores(const float* z, int T, int E, float* s, float* s_t, cudaStream_t stream) {
  if (T == 0 || E == 0) return LMOE_OK;
  if (ceil_div(T, 32) > 65535) return LMOE_ERR_UNSUPPORTED;  // grid rows
  const dim3 grid(static_cast<unsigned>(ceil_div(E, 32)), static_cast<unsigned>(ceil_div(T, 32)));
  return launch_pdl(scores_kernel, grid, 256, 0, stream, z, T, E, s, s_t) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_candidates(const float* z, int T, int E, int64_t stride_t, int64_t stride_e, int k,
                      float* cand, int64_t ldc, cudaStream_t stream) {
  if (E == 0 || k == 0) return LMOE_OK;
  const size_t smem =
      (TH_BINS + 32 + TH_CAND + (T <= TH_SMEM_MAX_T ? T : 0)) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(candidates_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  return launch_pdl(candidates_kernel, E, TH_THREADS, smem, stream, z, T, stride_t, stride_e, k,
                    cand, ldc) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

// Router backward.  Token t selected experts e_j with scores s_j = sigmoid(z[t, e_j]) and
// gates g_j = s_j / S, S the sum of the selected scores.  Given dg_j:
//   ds_j = (dg_j - sum_i g_i dg_i) / S,   dz[t, e_j] = ds_j s_j (1 - s_j),
// and dz[t, e] = 0 for the experts not selected.  One warp per token; the bf16 output row
// has ldo >= E columns, the ones past E zero.
__global__ void __launch_bounds__(256)
router_bwd_kernel(const float* __restrict__ z, int64_t ldz, const int32_t* __restrict__ idx,
                  const float* __restrict__ gate, const float* __restrict__ dgate, int T, int K,
                  __nv_bfloat16* __restrict__ dz, int ldo) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  __nv_bfloat16* row = dz + static_cast<size_t>(t) * ldo;
  for (int v = lane; v < ldo / 8; v += 32)
    reinterpret_cast<uint4*>(row)[v] = make_uint4(0u, 0u, 0u, 0u);
  float s = 0.0f, g = 0.0f, dg = 0.0f;
  int e = 0;
  if (lane < K) {
    const size_t j = static_cast<size_t>(t) * K + lane;
    e = __ldg(idx + j);
    s = score_sigmoid(__ldg(z + static_cast<size_t>(t) * ldz + e));
    g = __ldg(gate + j);
    dg = __ldg(dgate + j);
  }
  float S = s, dot = g * dg;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S += __shfl_xor_sync(0xffffffffu, S, o);
    dot += __shfl_xor_sync(0xffffffffu, dot, o);
  }
  __syncwarp();  // the zero fill above lands before the scattered entries
  if (lane < K) row[e] = __float2bfloat16_rn((dg - dot) / S * s * (1.0f - s));
}

int launch_router_bwd(const float* z, int64_t ldz, const int32_t* idx, const float* gate,
                      const float* dgate, int T, int K, __nv_bfloat16* dz, int ldo,
                      cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  if (K > 32 || ldo % 8 || (reinterpret_cast<uintptr_t>(dz) & 15)) return LMOE_ERR_UNSUPPORTED;
  return launch_pdl(router_bwd_kernel, static_cast<unsigned>(ceil_div(T, 8)), 256, 0, stream, z,
                    ldz, idx, gate, dgate, T, K, dz, ldo) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

// Checked mode: any non-finite value among p[0, n) sets DEVERR_NONFINITE.
__global__ void __launch_bounds__(256)
finite_check_kernel(const float* __restrict__ p, int64_t n, uint32_t* __restrict__ err) {
  pdl_wait();
  pdl_launch_dependents();
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    bad |= !isfinite(__ldg(p + i));
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(err, DEVERR_NONFINITE);
}

int launch_finite_check(const float* p, int64_t n, uint32_t* err, cudaStream_t stream) {
  if (n == 0) return LMOE_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  const int64_t blocks = ceil_div(n, 256);
  const unsigned grid = static_cast<unsigned>(blocks < 8 * sms ? blocks : 8 * sms);
  return launch_pdl(finite_check_kernel, grid, 256, 0, stream, p, n, err) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_transpose_f32(const float* in, int T, int E, float* out, cudaStream_t stream) {
  if (T == 0) return LMOE_OK;
  const dim3 grid(static_cast<unsigned>(ceil_div(E, 32)), static_cast<unsigned>(ceil_div(T, 32)));
  return launch_pdl(transpose_f32_kernel, grid, 256, 0, stream, in, T, E, out) == cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

}  // namespace lmoe
