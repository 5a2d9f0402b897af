// ep.cu -- expert-parallel dispatch and combine, packed and unpacked on one device.
//
// "Part 1 of Inside Kimi K3" (Towards AI article), Stable LatentMoE and communication
// passages: the routed experts live on different GPUs, each selected expert receives the
// token's vector, and the outputs travel back to be combined; projecting to the latent
// before the trip halves the bytes ("The 2.8-Trillion-Parameter Problem", Technical Details:
// 7168 -> 3584).  Here R ranks host the E experts in equal contiguous blocks.  Dispatch
// sends a token's row once to every rank that hosts at least one of its experts, with the
// mask of the token's slots served there; the pairs (token, rank) are laid out by rank, and
// by token within a rank.  The expert side returns one row per pair: the gate-weighted sum
// of its slots' outputs (an fp32 fused multiply-add chain in slot order, rounded to bf16);
// the source sums a token's returned rows in rank order in fp32.  The transfer itself (an
// all-to-all) is not part of this file: the buffers are what would cross the interconnect.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

constexpr int EP_WARPS = 8;

// masks[b * R + r] bit i <=> token 32 b + i sends its row to rank r.
__global__ void __launch_bounds__(EP_WARPS * 32)
ep_mask_kernel(const int32_t* __restrict__ idx, int T, int K, int per, int R,
               uint32_t* __restrict__ masks) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * EP_WARPS + (threadIdx.x >> 5);
  if (b * 32 >= T) return;
  const int t = b * 32 + lane;
  uint64_t rm = 0;
  if (t < T)
    for (int j = 0; j < K; ++j) {
      const int e = __ldg(idx + static_cast<size_t>(t) * K + j);
      if (e >= 0 && e < per * R) rm |= 1ull << (e / per);  // invalid indices go nowhere
    }
  for (int r = 0; r < R; ++r) {
    const uint32_t m = __ballot_sync(0xffffffffu, (rm >> r) & 1ull);
    if (lane == 0) masks[static_cast<size_t>(b) * R + r] = m;
  }
}

// base[b * R + r] = pairs of rank r in blocks < b; send_off = exclusive scan of the ranks'
// counts.  One CTA: warp w scans ranks w, w + 32, ...; each lane owns a strip of blocks.
__global__ void __launch_bounds__(1024)
ep_scan_kernel(const uint32_t* __restrict__ masks, int nb, int R, uint32_t* __restrict__ base,
               int32_t* __restrict__ send_off) {
  __shared__ int32_t count[64];
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int strip = (nb + 31) / 32;
  for (int r = warp; r < R; r += 32) {
    const int b0 = lane * strip, b1 = min(nb, b0 + strip);
    uint32_t s = 0;
    for (int b = b0; b < b1; ++b) s += __popc(masks[static_cast<size_t>(b) * R + r]);
    uint32_t incl = s;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    uint32_t run = incl - s;
    for (int b = b0; b < b1; ++b) {
      base[static_cast<size_t>(b) * R + r] = run;
      run += __popc(masks[static_cast<size_t>(b) * R + r]);
    }
    if (lane == 31) count[r] = static_cast<int32_t>(incl);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    for (int r = 0; r < R; ++r) {
      send_off[r] = acc;
      acc += count[r];
    }
    send_off[R] = acc;
  }
}

// Position of pair (t, r) in the send order.
__device__ __forceinline__ int ep_pair(const uint32_t* masks, const uint32_t* base,
                                       const int32_t* send_off, int R, int t, int r) {
  const int b = t >> 5, tl = t & 31;
  const size_t mb = static_cast<size_t>(b) * R + r;
  return __ldg(send_off + r) + static_cast<int>(__ldg(base + mb)) +
         __popc(__ldg(masks + mb) & ((1u << tl) - 1u));
}

// Slot j of token t (lanes j < K): the rank of its expert; the token's rank mask.
__device__ __forceinline__ uint64_t ep_ranks(const int32_t* idx, int t, int K, int per, int R,
                                             int lane, int* my_rank) {
  const int e = lane < K ? __ldg(idx + static_cast<size_t>(t) * K + lane) : -1;
  *my_rank = (e >= 0 && e < per * R) ? e / per : -1;
  uint64_t rm = *my_rank >= 0 ? 1ull << *my_rank : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rm |= __shfl_xor_sync(0xffffffffu, rm, o);
  return rm;
}

// Dispatch: one warp per token.
__global__ void __launch_bounds__(EP_WARPS * 32)
ep_dispatch_kernel(const int32_t* __restrict__ idx, int T, int K, int per, int R,
                   const uint32_t* __restrict__ masks, const uint32_t* __restrict__ base,
                   const int32_t* __restrict__ send_off, const uint4* __restrict__ rows, int W,
                   uint4* __restrict__ send_rows, int32_t* __restrict__ send_tok,
                   uint32_t* __restrict__ send_slots) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * EP_WARPS + (threadIdx.x >> 5);
  if (t >= T) return;
  int my_rank;
  uint64_t rm = ep_ranks(idx, t, K, per, R, lane, &my_rank);
  const int nv = W / 8;  // 16-byte vectors per row
  while (rm) {
    const int r = __ffsll(static_cast<long long>(rm)) - 1;
    rm &= rm - 1;
    const uint32_t slots = __ballot_sync(0xffffffffu, my_rank == r);
    const int p = ep_pair(masks, base, send_off, R, t, r);
    if (lane == 0) {
      send_tok[p] = t;
      send_slots[p] = slots;
    }
    if (rows)
      for (int v = lane; v < nv; v += 32)
        send_rows[static_cast<size_t>(p) * nv + v] = __ldg(rows + static_cast<size_t>(t) * nv + v);
  }
}

__device__ __forceinline__ void bf16x8_fma(float g, const uint4& u, float (&acc)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fmaf_rn(g, __uint_as_float(w[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = __fmaf_rn(g, __uint_as_float(w[i] & 0xFFFF0000u), acc[2 * i + 1]);
  }
}

// Combine, expert side: one warp per pair.
__global__ void __launch_bounds__(EP_WARPS * 32)
ep_combine_pack_kernel(const int32_t* __restrict__ send_off, int R, int pmax,
                       const int32_t* __restrict__ send_tok, const uint32_t* __restrict__ send_slots,
                       const int32_t* __restrict__ inv, const float* __restrict__ gate, int K,
                       const uint4* __restrict__ o, int W, uint4* __restrict__ part) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int p = blockIdx.x * EP_WARPS + (threadIdx.x >> 5);
  if (p >= pmax || p >= __ldg(send_off + R)) return;
  const int t = __ldg(send_tok + p);
  const uint32_t slots = __ldg(send_slots + p);
  const int nv = W / 8;
  for (int v = lane; v < nv; v += 32) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (uint32_t s = slots; s; s &= s - 1) {
      const int j = __ffs(s) - 1;
      const size_t tj = static_cast<size_t>(t) * K + j;
      bf16x8_fma(__ldg(gate + tj), __ldg(o + static_cast<size_t>(__ldg(inv + tj)) * nv + v), acc);
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    part[static_cast<size_t>(p) * nv + v] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Combine, source side: one warp per token; u = sum of its pairs' rows in rank order.
__global__ void __launch_bounds__(EP_WARPS * 32)
ep_combine_unpack_kernel(const int32_t* __restrict__ idx, int T, int K, int per, int R,
                         const uint32_t* __restrict__ masks, const uint32_t* __restrict__ base,
                         const int32_t* __restrict__ send_off, const uint4* __restrict__ part,
                         int W, float4* __restrict__ u) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * EP_WARPS + (threadIdx.x >> 5);
  if (t >= T) return;
  int my_rank;
  const uint64_t rm0 = ep_ranks(idx, t, K, per, R, lane, &my_rank);
  const int nv = W / 8;
  for (int v = lane; v < nv; v += 32) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (uint64_t rm = rm0; rm; rm &= rm - 1) {
      const int r = __ffsll(static_cast<long long>(rm)) - 1;
      const uint4 q = __ldg(part + static_cast<size_t>(ep_pair(masks, base, send_off, R, t, r)) * nv + v);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(w[i] << 16));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(w[i] & 0xFFFF0000u));
      }
    }
    float4* ur = u + static_cast<size_t>(t) * (W / 4) + 2 * v;
    ur[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    ur[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

size_t ep_workspace_bytes(int T, int R) {
  const size_t nb = static_cast<size_t>(ceil_div(T, 32));
  return 2 * nb * R * sizeof(uint32_t);
}

int launch_ep_dispatch(const int32_t* idx, int T, int K, int E, int R, const void* rows, int W,
                       void* send_rows, int32_t* send_off, int32_t* send_tok,
                       uint32_t* send_slots, void* ws, cudaStream_t stream) {
  const int nb = static_cast<int>(ceil_div(T, 32));
  const int per = E / R;
  uint32_t* masks = static_cast<uint32_t*>(ws);
  uint32_t* base = masks + static_cast<size_t>(nb) * R;
  if (launch_pdl(ep_mask_kernel, static_cast<unsigned>(ceil_div(nb, EP_WARPS)), EP_WARPS * 32, 0,
                 stream, idx, T, K, per, R, masks) != cudaSuccess ||
      launch_pdl(ep_scan_kernel, 1, 1024, 0, stream, static_cast<const uint32_t*>(masks), nb, R,
                 base, send_off) != cudaSuccess ||
      launch_pdl(ep_dispatch_kernel, static_cast<unsigned>(ceil_div(T, EP_WARPS)), EP_WARPS * 32, 0,
                 stream, idx, T, K, per, R, static_cast<const uint32_t*>(masks),
                 static_cast<const uint32_t*>(base), static_cast<const int32_t*>(send_off),
                 static_cast<const uint4*>(rows), W, static_cast<uint4*>(send_rows), send_tok,
                 send_slots) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

int launch_ep_combine(const int32_t* idx, int T, int K, int E, int R, const int32_t* send_off,
                      const int32_t* send_tok, const uint32_t* send_slots, const int32_t* inv,
                      const float* gate, const void* o, int W, void* part, float* u,
                      const void* ws, cudaStream_t stream) {
  const int nb = static_cast<int>(ceil_div(T, 32));
  const int per = E / R;
  const uint32_t* masks = static_cast<const uint32_t*>(ws);
  const uint32_t* base = masks + static_cast<size_t>(nb) * R;
  const int pmax = T * (K < R ? K : R);
  if (launch_pdl(ep_combine_pack_kernel, static_cast<unsigned>(ceil_div(pmax, EP_WARPS)),
                 EP_WARPS * 32, 0, stream, send_off, R, pmax, send_tok, send_slots, inv, gate, K,
                 static_cast<const uint4*>(o), W, static_cast<uint4*>(part)) != cudaSuccess ||
      launch_pdl(ep_combine_unpack_kernel, static_cast<unsigned>(ceil_div(T, EP_WARPS)),
                 EP_WARPS * 32, 0, stream, idx, T, K, per, R, masks, base, send_off,
                 static_cast<const uint4*>(part), W, reinterpret_cast<float4*>(u)) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

}  // namespace lmoe
