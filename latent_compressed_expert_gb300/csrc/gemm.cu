// gemm.cu -- persistent, warp-specialised bf16 GEMM on the 5th-generation tensor cores.
//
//   C[M, N] = A[M, Kd] . B[N, Kd]^T      (A and B K-major, fp32 accumulation in TMEM)
//
// One CTA per SM walks a list of 128 x BN output tiles (BN = 128 or 256):
//   warp 0      TMA producer: 64-wide K slices of A (128 rows) and B (BN rows) into a ring
//               of shared-memory stages, completing on per-stage "full" mbarriers;
//   warp 1      allocates 2 x BN TMEM columns (two accumulators) and issues
//               tcgen05.mma (M=128, N=BN, K=16) from one thread; tcgen05.commit frees each
//               stage ("empty") and announces each finished accumulator ("tmem_full");
//   warps 2-5   epilogue: tcgen05.ld of 32 columns at a time, the fused operation (plain
//               bf16 / fp32 store, SiTU-GLU on interleaved gate/value columns, residual add),
//               then release the accumulator ("tmem_empty") so the MMA of the tile after
//               next can start while this one is written out.
// Tile pairs (MT = 2): a CTA computes two 128-row M-tiles that share each B stage, two MMAs
// per K-step into the two halves of TMEM (one accumulator, drained before the next pair),
// for long dense reductions: half the B bytes per FLOP.
// Grouped-K mode (the backward's weight gradients): `groups` independent products, each a
// reduction over its own range of rows of token-major operands, which the MMA reads as
// MN-major tiles (64 x 64 TMA boxes); A's rows past a group's end are zeroed in shared
// memory before its last K-block's MMAs.
// This kernel serves the dense contractions (x-side GEMM, router, output GEMM, the
// backward's dense GEMMs and weight gradients); the routed experts' forward and dgrad GEMMs
// are in gemm_grouped.cu.
//
// Every wait is bounded (globaltimer); on time-out a role records an error bit in global
// memory, raises a shared abort flag that makes the other roles give up too, waits for
// its in-flight copies and MMAs, and the CTA frees its TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace lmoe {

// MT: 128-row M-tiles per CTA.  MT = 2 computes a 256 x BN tile pair that shares each B
// stage: two MMAs per K-step into the two halves of TMEM, half the B bytes per FLOP, so the
// same shared memory covers a longer load latency.  Its single accumulator is drained
// before the next pair starts, so it serves long reductions (dense mode only).
// TMEM is allocated in powers of two columns (32 at least).
constexpr int tmem_alloc_cols(int cols) {
  int n = 32;
  while (n < cols) n *= 2;
  return n;
}

// BN = 224 serves N = 896 (the router over 896 experts) in four whole column tiles.
template <int BN, int MT>
struct GemmCfg {
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K * 2;  // one 128-row M-tile
  static constexpr int B_BYTES = BN * BLOCK_K * 2;
  static constexpr int STAGE_BYTES = MT * A_BYTES + B_BYTES;
  static constexpr int STAGES = BN >= 224 ? (MT == 2 ? 3 : 4) : (MT == 2 ? 4 : 6);
  static constexpr int ACC = MT == 2 ? 1 : 2;  // accumulator buffers of MT x BN columns
  static constexpr int TMEM_COLS = tmem_alloc_cols(2 * BN);
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 6;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  // grouped-K epilogue staging: two buffers of 32 rows x 32 fp32 per epilogue warp, 1024-byte
  // aligned (their 16-byte chunks are placed with the 128-byte swizzle that the tensor stores
  // writing them out apply)
  static constexpr int EPI_OFF = (MISC_OFF + 16 + 1023) / 1024 * 1024;
  static constexpr int EPI_BYTES = MT == 1 ? 2 * 4 * 32 * 32 * 4 : 0;
  static constexpr int SMEM_BYTES = EPI_OFF + EPI_BYTES + 1024;  // + slack for 1024 alignment
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BLOCK_M, BN);
  static constexpr uint32_t IDESC_MN = ptx::idesc_bf16_f32_mn(BLOCK_M, BN);
  static constexpr int BOX_BYTES = 64 * BLOCK_K * 2;  // one 64 x 64 MN-major TMA box
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "tiles must stay 1024-aligned");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

constexpr int GEMM_THREADS = 192;
constexpr int GEMM_PAIR_MIN_K = 2048;  // reduction length from which tile pairs are used
constexpr int SPLITK_MIN_KB = 4;       // K-blocks per split-K slice at least
constexpr int RASTER_GROUP_M = 16;

struct TileCoord {
  int a_row;    // first row of A (and of the output) of this tile
  int row_end;  // rows >= row_end are not part of this problem
  int b_row;    // first row of B
  int n0;       // first output column
  int grp;      // grouped-K mode: the group; else 0
  int k0;       // first K index (column of A and B; grouped-K: their first row) reduced over
  int nk;       // 64-wide K-blocks reduced over
  int klen;     // grouped-K: rows in the group (the last K-block may be partial)
};

template <int BN, int TM = BLOCK_M>  // TM: rows of an M-tile (of a tile pair)
__device__ __forceinline__ TileCoord decode_tile(const GemmArgs& g, int nt, int mt, int tile) {
  int kgroup = 0;
  if (g.groups > 0 || g.ksplit > 1) {  // groups (or split-K slices) outermost, then the raster
    kgroup = tile / (mt * nt);
    tile -= kgroup * mt * nt;
  }
  // groups of RASTER_GROUP_M row tiles sweep all column tiles, rows fastest, so the CTAs in
  // flight share a few A row-panels and B column-panels in L2
  const int span = RASTER_GROUP_M * nt;
  const int grp = tile / span;
  const int first_m = grp * RASTER_GROUP_M;
  const int gm = min(RASTER_GROUP_M, mt - first_m);
  const int local = tile - grp * span;
  const int m = first_m + local % gm;
  const int n = local / gm;
  TileCoord c;
  c.a_row = m * TM;
  c.row_end = g.M;
  c.b_row = n * BN;
  c.n0 = n * BN;
  c.grp = kgroup;
  if (g.groups > 0) {
    c.k0 = __ldg(g.kseg + kgroup);
    c.klen = __ldg(g.kseg + kgroup + 1) - c.k0;
    c.nk = (c.klen + BLOCK_K - 1) / BLOCK_K;
  } else if (g.ksplit > 1) {  // slice kgroup of the K-blocks (the launcher leaves none empty)
    const int nkb = g.Kd / BLOCK_K;
    const int per = (nkb + g.ksplit - 1) / g.ksplit;
    c.k0 = kgroup * per * BLOCK_K;
    c.nk = min(per, nkb - kgroup * per);
    c.klen = c.nk * BLOCK_K;
  } else {
    c.k0 = 0;
    c.klen = g.Kd;
    c.nk = g.Kd / BLOCK_K;
  }
  return c;
}

__device__ __forceinline__ void raise_error(const GemmArgs& g, volatile int* abort_flag,
                                            uint32_t code) {
  *abort_flag = 1;
  atomicOr(g.err, code);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u && ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  uint4 w;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  return w;
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) o[q] = pack8_bf16(v + 8 * q);
}

// SiTU-GLU: silu(c tanh(g/c)) * c tanh(v/c).  ("The 2.8-Trillion-Parameter Problem",
// Technical Details / Stabilization Mechanisms: gate and value smoothly capped to about
// +-100, SwiGLU-like near zero; the tanh cap is this library's reading of "smoothly caps".)
__device__ __forceinline__ float situ(float g, float v, float c, float inv_c) {
  const float gc = c * ptx::tanh_approx(g * inv_c);
  const float vc = c * ptx::tanh_approx(v * inv_c);
  const float sg = __fdividef(gc, 1.0f + __expf(fminf(-gc, 80.0f)));
  return sg * vc;
}

// 32 accumulator columns = 16 gate (0..15) + the matching 16 value (16..31) -> 16 outputs.
__device__ __forceinline__ void store_situ16(__nv_bfloat16* dst, const float (&v)[32], float c,
                                             float inv_c) {
  float o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = situ(v[i], v[16 + i], c, inv_c);
  uint4* p = reinterpret_cast<uint4*>(dst);
  p[0] = pack8_bf16(o);
  p[1] = pack8_bf16(o + 8);
}

__device__ __forceinline__ void epilogue_store(const GemmArgs& g, int row, int col0,
                                               float (&v)[32], float c, float inv_c) {
  const size_t r = static_cast<size_t>(row);
  switch (g.epi) {
    case EPI_BF16:
      store_bf16x32(g.out0 + r * g.ld0 + col0, v);
      break;
    case EPI_F32: {
      if (g.col_bias) {
        const float4* bp = reinterpret_cast<const float4*>(g.col_bias + col0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 b = __ldg(bp + q);
          v[4 * q] += b.x;
          v[4 * q + 1] += b.y;
          v[4 * q + 2] += b.z;
          v[4 * q + 3] += b.w;
        }
      }
      float4* o = reinterpret_cast<float4*>(g.outf + r * g.ldf + col0);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      if (g.outf_t) {  // a warp's 32 rows are consecutive: 128-byte runs per column
#pragma unroll
        for (int i = 0; i < 32; ++i) g.outf_t[static_cast<size_t>(col0 + i) * g.ldt + r] = v[i];
      }
      break;
    }
    case EPI_SITU:
      if (g.pre) store_bf16x32(g.pre + r * g.ldp + col0, v);
      store_situ16(g.out1 + r * g.ld1 + col0 / 2, v, c, inv_c);
      break;
    case EPI_SPLIT:
      if (col0 < g.split) {
        store_bf16x32(g.out0 + r * g.ld0 + col0, v);
      } else {
        if (g.pre) store_bf16x32(g.pre + r * g.ldp + (col0 - g.split), v);
        store_situ16(g.out1 + r * g.ld1 + (col0 - g.split) / 2, v, c, inv_c);
      }
      break;
    case EPI_RESID:
    default: {
      if (g.addf) {
        const float4* ap = reinterpret_cast<const float4*>(g.addf + r * g.lda + col0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 a = __ldg(ap + q);
          v[4 * q] += a.x;
          v[4 * q + 1] += a.y;
          v[4 * q + 2] += a.z;
          v[4 * q + 3] += a.w;
        }
      }
      if (g.resid) {
        const uint4* rp = reinterpret_cast<const uint4*>(g.resid + r * g.ldr + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 raw = __ldg(rp + q);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            v[8 * q + 2 * i] += f.x;
            v[8 * q + 2 * i + 1] += f.y;
          }
        }
      }
      if (g.outf) {  // the value before its rounding to bf16
        float4* o = reinterpret_cast<float4*>(g.outf + r * g.ldf + col0);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      store_bf16x32(g.out0 + r * g.ld0 + col0, v);
      break;
    }
  }
}

// EPI_RESID with the chunk's residual already loaded (raw bf16, 4 x 16 bytes): the dense
// epilogue loads chunk i + 1's residual before it waits on chunk i's accumulator columns, so
// the global-load latency is paid once per tile rather than once per 32-column chunk.
__device__ __forceinline__ void store_resid_prefetched(const GemmArgs& g, int row, int col0,
                                                       float (&v)[32], const uint4 (&rv)[4]) {
  const size_t r = static_cast<size_t>(row);
  if (g.addf) {
    const float4* ap = reinterpret_cast<const float4*>(g.addf + r * g.lda + col0);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 a = __ldg(ap + q);
      v[4 * q] += a.x;
      v[4 * q + 1] += a.y;
      v[4 * q + 2] += a.z;
      v[4 * q + 3] += a.w;
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&rv[q]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[8 * q + 2 * i] += f.x;
      v[8 * q + 2 * i + 1] += f.y;
    }
  }
  if (g.outf) {  // the value before its rounding to bf16
    float4* o = reinterpret_cast<float4*>(g.outf + r * g.ldf + col0);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
  store_bf16x32(g.out0 + r * g.ld0 + col0, v);
}

// Last, partly valid 32-column slice (plain stores only; the GLU modes need whole slices).
__device__ __forceinline__ void epilogue_store_partial(const GemmArgs& g, int row, int col0,
                                                   int ncols, const float (&v)[32]) {
  const size_t r = static_cast<size_t>(row);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (i >= ncols) break;
    const int col = col0 + i;
    if (g.epi == EPI_F32) {
      const float t = g.col_bias ? v[i] + __ldg(g.col_bias + col) : v[i];
      g.outf[r * g.ldf + col] = t;
      if (g.outf_t) g.outf_t[static_cast<size_t>(col) * g.ldt + r] = t;
    } else if (g.epi == EPI_BF16) {
      g.out0[r * g.ld0 + col] = __float2bfloat16_rn(v[i]);
    } else if (g.epi == EPI_RESID) {
      float t = v[i];
      if (g.addf) t += g.addf[r * g.lda + col];
      if (g.resid) t += __bfloat162float(g.resid[r * g.ldr + col]);
      if (g.outf) g.outf[r * g.ldf + col] = t;
      g.out0[r * g.ld0 + col] = __float2bfloat16_rn(t);
    }
  }
}

// RP: the residual epilogue with its residual prefetched one chunk ahead (the output GEMM);
// a separate instantiation, so that the other epilogues keep their own code.
template <int BN, int MT, bool RP>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmO, const GemmArgs g) {
  using C = GemmCfg<BN, MT>;
  constexpr int TM = BLOCK_M * MT;
  if constexpr (MT != 1 || BN % 64 != 0) {
    // tile pairs and 224-wide tiles serve the dense mode only (grouped-K loads B in 64-row
    // boxes); the launcher never does this
    if (g.groups > 0) {
      if (threadIdx.x == 0) atomicOr(g.err, DEVERR_BAD_INDEX);
      return;
    }
  }
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* stall = drain + 1;  // never arrived on (fault-injection hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = (g.N + BN - 1) / BN;
  const int mt_dense = (g.M + TM - 1) / TM;
  const int total =
      mt_dense * nt * (g.groups > 0 ? g.groups : 1) * (g.ksplit > 1 ? g.ksplit : 1);
  const uint64_t limit = g.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 128);
    }
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(stall, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // from here on: the previous kernel's outputs are visible
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileCoord tc = decode_tile<BN, TM>(g, nt, mt_dense, tile);
        for (int kb = 0; kb < tc.nk; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, limit)) {
            raise_error(g, abort_flag, DEVERR_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * C::STAGE_BYTES;
          ptx::mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          if (g.groups > 0) {
            // MN-major: 64 K rows of 64-column boxes (rows past the operand are zero-filled)
            const int krow = tc.k0 + kb * BLOCK_K;
#pragma unroll
            for (int i = 0; i < BLOCK_M / 64; ++i)
              ptx::tma_load_2d(sa + i * C::BOX_BYTES, &tmA, &full[s], tc.a_row + 64 * i, krow);
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              ptx::tma_load_2d(sa + C::A_BYTES + i * C::BOX_BYTES, &tmB, &full[s],
                               tc.b_row + 64 * i, krow);
          } else {
#pragma unroll
            for (int i = 0; i < MT; ++i)  // rows past M are zero-filled
              ptx::tma_load_2d(sa + i * C::A_BYTES, &tmA, &full[s], tc.k0 + kb * BLOCK_K,
                               tc.a_row + i * BLOCK_M);
            ptx::tma_load_2d(sa + MT * C::A_BYTES, &tmB, &full[s], tc.k0 + kb * BLOCK_K,
                             tc.b_row);
          }
        }
      }
      // every issued copy must land before the CTA may exit
      const uint32_t first = it > static_cast<uint32_t>(C::STAGES) ? it - C::STAGES : 0u;
      for (uint32_t j = first; j < it; ++j) {
        if (!wait_drain(&full[j % C::STAGES], (j / C::STAGES) & 1u, limit)) {
          raise_error(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
          break;
        }
      }
    }
  } else if (warp == 1 && g.groups > 0) {
    // ------------------------------------------------------------ MMA issuer, grouped-K:
    // the whole warp waits; in a group's last K-block it zeroes A's rows past the group
    // (another group's rows, or TMA fill), then one lane issues the MMAs
    uint32_t it = 0;
    int lt = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++lt) {
      const int acc = lt & 1;
      const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, limit))) {
        if (lane == 0) raise_error(g, abort_flag, DEVERR_TIMEOUT_MMA);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      const TileCoord tc = decode_tile<BN, TM>(g, nt, mt_dense, tile);
      for (int kb = 0; kb < tc.nk; ++kb, ++it) {
        const int s = static_cast<int>(it % C::STAGES);
        const uint32_t ph = (it / C::STAGES) & 1u;
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&full[s], ph, abort_flag, limit))) {
          if (lane == 0) raise_error(g, abort_flag, DEVERR_TIMEOUT_MMA);
          ok = false;
          break;
        }
        uint8_t* sa = smem + s * C::STAGE_BYTES;
        const int valid = tc.klen - kb * BLOCK_K;  // K rows of this block inside the group
        if (valid < BLOCK_K) {
          // a K row is one 128-byte line of each A box (the swizzle permutes within it)
          const int per_box = (BLOCK_K - valid) * 8;  // 16-byte pieces
          for (int i = lane; i < (BLOCK_M / 64) * per_box; i += 32) {
            const int box = i / per_box, rem = i - box * per_box;
            *reinterpret_cast<uint4*>(sa + box * C::BOX_BYTES + valid * 128 + rem * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          ptx::fence_proxy_async_smem();  // the zeros are visible to the tensor cores
        }
        __syncwarp();
        if (lane == 0) {
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(sa);
          const uint32_t b0 = a0 + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < BLOCK_K / 16; ++k)  // 16 K rows = two 1024-byte atoms
            ptx::umma_bf16(d_tmem, ptx::smem_desc_sw128_mn(a0 + k * 2048, C::BOX_BYTES),
                           ptx::smem_desc_sw128_mn(b0 + k * 2048, C::BOX_BYTES), C::IDESC_MN,
                           (kb | k) != 0 ? 1u : 0u);
          ptx::umma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) ptx::umma_commit(&tfull[acc]);
    }
    if (lane == 0) {
      // all MMAs issued by this thread complete before TMEM is released
      ptx::umma_commit(drain);
      if (!wait_drain(drain, 0u, limit)) raise_error(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      uint32_t it = 0;
      int lt = 0;
      bool stalled = false;
      if (g.inject_stall && !ptx::mbar_wait(stall, 0u, abort_flag, limit)) {
        raise_error(g, abort_flag, DEVERR_TIMEOUT_MMA);
        stalled = true;
      }
      for (int tile = blockIdx.x; !stalled && tile < total; tile += gridDim.x, ++lt) {
        const int acc = C::ACC == 2 ? (lt & 1) : 0;
        const uint32_t aph = C::ACC == 2 ? (static_cast<uint32_t>(lt >> 1) & 1u)
                                         : (static_cast<uint32_t>(lt) & 1u);
        if (!ptx::mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, limit)) {
          raise_error(g, abort_flag, DEVERR_TIMEOUT_MMA);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const int nkt =
            g.ksplit > 1 ? decode_tile<BN, TM>(g, nt, mt_dense, tile).nk : g.Kd / BLOCK_K;
        bool ok = true;
        for (int kb = 0; kb < nkt; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&full[s], ph, abort_flag, limit)) {
            raise_error(g, abort_flag, DEVERR_TIMEOUT_MMA);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + MT * C::A_BYTES;
#pragma unroll
          for (int k = 0; k < BLOCK_K / 16; ++k)
#pragma unroll
            for (int i = 0; i < MT; ++i)  // M-tile i accumulates into TMEM columns i*BN..
              ptx::umma_bf16(d_tmem + static_cast<uint32_t>(i * BN),
                             ptx::smem_desc_sw128(sa + i * C::A_BYTES + k * 32),
                             ptx::smem_desc_sw128(sb + k * 32), C::IDESC,
                             (kb | k) != 0 ? 1u : 0u);
          ptx::umma_commit(&empty[s]);
        }
        if (!ok) break;
        ptx::umma_commit(&tfull[acc]);
      }
      // all MMAs issued by this thread complete before TMEM is released
      ptx::umma_commit(drain);
      if (!wait_drain(drain, 0u, limit)) raise_error(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // this warp's two staging buffers (grouped-K): buffer b at EPI_OFF + (4 b + q) * 4 KB
    float* stage0 = reinterpret_cast<float*>(smem + C::EPI_OFF) + q * 32 * 32;
    int nst = 0;  // grouped-K chunks this warp has handed to tensor stores
    const float c = g.c, inv_c = 1.0f / g.c;
    int lt = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++lt) {
      const int acc = C::ACC == 2 ? (lt & 1) : 0;
      const uint32_t aph = C::ACC == 2 ? (static_cast<uint32_t>(lt >> 1) & 1u)
                                       : (static_cast<uint32_t>(lt) & 1u);
      const bool got = ptx::mbar_wait(&tfull[acc], aph, abort_flag, limit);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) raise_error(g, abort_flag, DEVERR_TIMEOUT_EPILOGUE);
        break;
      }
      ptx::tc_fence_after();
      const TileCoord tc = decode_tile<BN, TM>(g, nt, mt_dense, tile);
      // the M-tiles of the tile (two for a tile pair), at TMEM columns (acc + h) * BN
#pragma unroll 1
      for (int h = 0; h < MT; ++h) {
        const int row = tc.a_row + h * BLOCK_M + q * 32 + lane;
        const bool row_ok = row < tc.row_end;
        const int orow =
            (g.groups > 0 && row_ok) ? (g.row_map ? __ldg(g.row_map + row) : row) : 0;
        // grouped-K with tensor stores: the warp's rows 0..15 and 16..31 must each land on
        // 16 consecutive output rows (the gate/value de-interleave keeps 16-row runs)
        const int orun0 = __shfl_sync(0xffffffffu, orow, 0);
        const int orun1 = __shfl_sync(0xffffffffu, orow, 16);
        const bool tma_rows = g.out_tma && __all_sync(0xffffffffu, row_ok &&
            orow == (lane < 16 ? orun0 + lane : orun1 + lane - 16));
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>((acc + h) * BN);
        // Residual epilogue over whole 32-column chunks: chunk ch + 1's residual is loaded
        // before chunk ch's accumulator columns are read (the launcher sets RP only for
        // this case, so the condition is warp-uniform; the tcgen05.ld is executed by every
        // lane, the global accesses by the rows inside M).
        if constexpr (RP) {
          const uint4* rrow = reinterpret_cast<const uint4*>(
              g.resid + static_cast<size_t>(row_ok ? row : 0) * g.ldr + tc.n0);
          uint4 rnext[4];
          if (row_ok) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) rnext[q4] = __ldg(rrow + q4);
          }
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ++ch) {
            uint4 rcur[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) rcur[q4] = rnext[q4];
            if (row_ok && ch + 1 < BN / 32) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) rnext[q4] = __ldg(rrow + 4 * (ch + 1) + q4);
            }
            float v[32];
            ptx::tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(ch * 32), v);
            if (row_ok) store_resid_prefetched(g, row, tc.n0 + ch * 32, v, rcur);
          }
          continue;
        }
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
          const int col0 = tc.n0 + ch * 32;
          if (col0 >= g.N) break;  // uniform across the warp
          float v[32];
          if (g.groups > 0) {
            // grouped-K: an empty reduction range is a zero product
            if (tc.nk > 0) {
              ptx::tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(ch * 32), v);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            }
            // Through this warp's staging buffer (16-byte chunks XOR-swizzled by row): either
            // two tensor stores of 16 rows x 32 columns issued by lane 0, or store
            // instructions that each write four whole 128-byte row segments.
            float* stage = stage0 + (nst & 1) * (4 * 32 * 32);
            if (tma_rows || nst > 0) {
              // the store that last read this buffer (two chunks back) is done reading it;
              // before thread stores, every earlier tensor store is
              if (lane == 0) {
                if (tma_rows)
                  ptx::bulk_wait_group_read<1>();
                else
                  ptx::bulk_wait_group_read<0>();
              }
              __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              reinterpret_cast<float4*>(stage + lane * 32)[j ^ (lane & 7)] =
                  make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            if (tma_rows) {
              ptx::fence_proxy_async_smem();  // the rows, visible to the tensor store
              __syncwarp();
              if (lane == 0) {  // columns past N and rows past M are clipped by the map
                ptx::tma_store_3d(&tmO, stage, col0, orun0, tc.grp);
                ptx::tma_store_3d(&tmO, stage + 16 * 32, col0, orun1, tc.grp);
                ptx::bulk_commit_group();
              }
              ++nst;
              continue;
            }
            __syncwarp();
            const int nvalid = min(32, g.N - col0);  // a multiple of 16
            const int c4 = lane & 7;
            float* og = g.outf + tc.grp * g.group_stride + col0 + 4 * c4;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int r = 4 * it + (lane >> 3);
              const int orow_r = __shfl_sync(0xffffffffu, orow, r);
              const bool ok_r = __shfl_sync(0xffffffffu, row_ok ? 1 : 0, r) != 0;
              if (ok_r && 4 * c4 < nvalid)
                *reinterpret_cast<float4*>(og + static_cast<size_t>(orow_r) * g.ldf) =
                    reinterpret_cast<const float4*>(stage + r * 32)[c4 ^ (r & 7)];
            }
            __syncwarp();
            continue;
          }
          ptx::tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(ch * 32), v);
          if (g.ksplit > 1) {  // split-K: this slice's fp32 partial sums
            if (row_ok) {
              float4* pp = reinterpret_cast<float4*>(
                  g.partial + (static_cast<size_t>(tc.grp) * g.M + row) * g.N + col0);
              const int nv4 = min(32, g.N - col0) / 4;  // N is a multiple of 16
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                if (q4 < nv4)
                  pp[q4] = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
            }
            continue;
          }
          if (row_ok) {
            if (col0 + 32 <= g.N)
              epilogue_store(g, row, col0, v, c, inv_c);
            else
              epilogue_store_partial(g, row, col0, g.N - col0, v);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[acc]);
    }
    // the tensor stores complete before the CTA leaves (they read its shared memory)
    if (lane == 0 && nst > 0) ptx::bulk_wait_group_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// Split-K: out = epilogue(sum over the slices of partial[s, row, :]), each chunk's slices
// added in a fixed order (deterministic).  Two forms:
//   WARP = false: one thread per row and 32-column chunk adds the slices in order and applies
//     the epilogue; for a few slices and many chunks.
//   WARP = true: one warp per chunk.  Lane l loads 16 bytes (float4 l % 8 of the chunk) of
//     every fourth slice from l / 8, so a warp has 32 loads in flight; a fixed shuffle tree
//     adds the four lanes of each float4, and lane 0 gathers the chunk and applies the
//     epilogue.  For many slices and few chunks.
constexpr int SPLITK_WARP_MIN = 7;  // slices from which the warp form is used

template <bool WARP>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const GemmArgs g) {
  pdl_wait();
  pdl_launch_dependents();
  const float c = g.c, inv_c = 1.0f / g.c;
  const int lane = threadIdx.x & 31;
  const int nch = (g.N + 31) / 32;
  const int64_t n = static_cast<int64_t>(g.M) * nch;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t w = WARP ? (tid >> 5) : tid; w < n; w += WARP ? (stride >> 5) : stride) {
    const int row = static_cast<int>(w / nch);
    const int col0 = static_cast<int>(w % nch) * 32;
    const int nv4 = min(32, g.N - col0) / 4;  // N is a multiple of 16
    float v[32];
    if constexpr (WARP) {  // w is warp-uniform here
      const int q4 = lane & 7;
      float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (q4 < nv4) {
        for (int sl = lane >> 3; sl < g.ksplit; sl += 4) {
          const float4 t = __ldg(reinterpret_cast<const float4*>(
              g.partial + (static_cast<size_t>(sl) * g.M + row) * g.N + col0) + q4);
          a.x += t.x;
          a.y += t.y;
          a.z += t.z;
          a.w += t.w;
        }
      }
#pragma unroll
      for (int o = 8; o <= 16; o <<= 1) {
        a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
        a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
        a.z += __shfl_xor_sync(0xffffffffu, a.z, o);
        a.w += __shfl_xor_sync(0xffffffffu, a.w, o);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[4 * q] = __shfl_sync(0xffffffffu, a.x, q);
        v[4 * q + 1] = __shfl_sync(0xffffffffu, a.y, q);
        v[4 * q + 2] = __shfl_sync(0xffffffffu, a.z, q);
        v[4 * q + 3] = __shfl_sync(0xffffffffu, a.w, q);
      }
      if (lane != 0) continue;
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      for (int sl = 0; sl < g.ksplit; ++sl) {
        const float4* pp = reinterpret_cast<const float4*>(
            g.partial + (static_cast<size_t>(sl) * g.M + row) * g.N + col0);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          if (q4 < nv4) {
            const float4 t = __ldg(pp + q4);
            v[4 * q4] += t.x;
            v[4 * q4 + 1] += t.y;
            v[4 * q4 + 2] += t.z;
            v[4 * q4 + 3] += t.w;
          }
        }
      }
    }
    if (nv4 == 8)
      epilogue_store(g, row, col0, v, c, inv_c);
    else
      epilogue_store_partial(g, row, col0, 4 * nv4, v);
  }
}

// ------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// fp32 output of `groups` row-major [rows, cols] matrices (row stride ld, group stride gstride
// elements) as a 3-D tensor with boxes of 32 columns x 16 rows, 128-byte swizzled.
static bool make_tmap_f32_out(CUtensorMap* m, const float* ptr, int cols, int rows, int groups,
                              int ld, long long gstride) {
  auto enc = tmap_encoder();
  if (!enc || !ptr || rows <= 0 || cols <= 0 || groups <= 0 ||
      (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0 || ld % 4 != 0 || ld < cols)
    return false;
  const long long gs = groups > 1 ? gstride : static_cast<long long>(rows) * ld;
  if (gs % 4 != 0 || gs < static_cast<long long>(rows) * ld) return false;
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(groups)};
  const cuuint64_t gstr[2] = {static_cast<cuuint64_t>(ld) * 4, static_cast<cuuint64_t>(gs) * 4};
  const cuuint32_t box[3] = {32, 16, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), gdim,
                         gstr, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 output rows [rows, cols] (row stride ld) for tensor stores of 32 x 32 boxes whose 64-byte
// rows hold their 16-byte pieces XOR-swizzled by (row / 2) % 4 (the 64-byte swizzle).
bool make_tmap_bf16_out32(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                          uint64_t ld) {
  auto enc = tmap_encoder();
  if (!enc || rows == 0 || cols == 0 || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0 ||
      (ld * 2) % 16 != 0 || ld < cols)
    return false;
  const cuuint64_t gdim[2] = {cols, rows};
  const cuuint64_t gstride[1] = {ld * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim,
                         gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                    uint32_t box_rows) {
  auto enc = tmap_encoder();
  if (!enc || rows == 0 || cols == 0 || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0 ||
      (ld * 2) % 16 != 0)
    return false;
  const cuuint64_t gdim[2] = {cols, rows};
  const cuuint64_t gstride[1] = {ld * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BLOCK_K), box_rows};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim,
                         gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------------------
// Dense GEMM over an SM pair (tcgen05 cta_group::2).
//
// A cluster of two CTAs on two SMs computes a 256 x 256 output tile with MMAs of M = 256,
// N = 256 issued by rank 0: rank r holds A's rows 128 r .. 128 r + 127 of the tile and B's
// rows (output columns) 128 r .. 128 r + 127, and each MMA reads both CTAs' shared memory at
// the same offsets.  Each CTA's TMEM receives its 128 output rows x all 256 columns, so an
// accumulator set takes 256 columns and two fit: the epilogue drains tile i while the MMAs
// of tile i + 1 run.  Per K-block an SM stages 16 KB of A and 16 KB of B for its 128 x 256 x
// 64 share of the MMA -- the bytes per FLOP of a one-SM tile pair, whose accumulators take all
// of TMEM and are drained while no MMA runs (12-16 % of the prefill GEMMs' time).  The
// epilogue is the one-SM kernel's, row by row.
//
// Synchronisation (every wait bounded): full[s] of rank 0 completes when both CTAs' TMA bytes
// for stage s have landed (rank 0's producer expects both; rank 1's copies complete on rank
// 0's barrier); empty[s] and tfull[a] of both CTAs get one arrival each from rank 0's commits
// (multicast); tempty[a] of rank 0 gets one arrival per epilogue warp of both CTAs; cluster
// barriers bracket set-up and teardown, so that neither CTA leaves while its peer may still
// signal its barriers or read its shared memory.
// The grouped-K epilogue writes its fp32 output with tensor stores from the staging buffers
// (else with store instructions from its threads).
constexpr bool GEMM_WGRAD_TMA_STORE = true;
constexpr bool GEMM_WGRAD_SM_PAIR = true;  // single-range weight gradients over SM pairs
constexpr int GEMM_PAIR_STAGES = 7;
constexpr bool GEMM_SM_PAIR = true;  // the tile-pair GEMMs run over SM pairs

template <int BN_>
struct GemmPairCfg {
  static constexpr int BN = BN_;                          // output columns per cluster tile
  static constexpr int TM = 2 * BLOCK_M;                  // output rows per cluster tile
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K * 2;   // this CTA's 128 rows of A
  static constexpr int B_BYTES = (BN / 2) * BLOCK_K * 2;  // this CTA's 128 rows of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 32 KB (BN = 256) or 30 KB
  static constexpr int STAGES = GEMM_PAIR_STAGES;
  static constexpr int TMEM_COLS = 512;                   // two accumulator sets of BN columns
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 6;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack for 1024 alignment
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(TM, BN);
  static constexpr uint32_t IDESC_MN = ptx::idesc_bf16_f32_mn(TM, BN);
  static constexpr int BOX_BYTES = 64 * BLOCK_K * 2;     // one 64 x 64 MN-major TMA box
  static_assert(BN % 32 == 0 && BN <= 256 && 2 * BN <= TMEM_COLS, "two accumulator sets fit TMEM");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "tiles must stay 1024-aligned");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// BN: 256, or 224 (the router over 896 experts: four whole column tiles).  RP: the residual
// epilogue with its residual prefetched one chunk ahead (the output GEMM).  MN: a weight
// gradient C = A^T B over all g.kfull rows of token-major A [kfull, M] and B [kfull, N], read
// as MN-major operands in 64 x 64 boxes (rows past kfull are zero-filled by TMA); fp32 output
// at row g.row_map[r] (or r).
template <int BN, bool RP, bool MN = false>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmArgs g) {
  using C = GemmPairCfg<BN>;
  static_assert(!MN || (BN == 256 && !RP), "MN-major operands: 256-wide tiles, fp32 output");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* stall = drain + 1;  // never arrived on (fault-injection hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const uint32_t rank = ptx::cluster_ctarank();  // rank 0 issues the MMAs
  const bool lead = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = (g.N + C::BN - 1) / C::BN;
  const int mt = (g.M + C::TM - 1) / C::TM;
  const int total = mt * nt;
  const int nk = MN ? (g.kfull + BLOCK_K - 1) / BLOCK_K : g.Kd / BLOCK_K;
  const uint64_t limit = g.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);  // rank 0's producer; the bytes come from both CTAs
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 2 * 4);  // lane 0 of the four epilogue warps of each CTA
    }
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(stall, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other's
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // from here on: the previous kernel's outputs are visible
  pdl_launch_dependents();
  const int cid = static_cast<int>(ptx::cluster_id_x());
  const int ncl = static_cast<int>(ptx::ncluster_x());

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both ranks)
      uint32_t it = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl) {
        const TileCoord tc = decode_tile<C::BN, C::TM>(g, nt, mt, tile);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, limit)) {
            raise_error(g, abort_flag, DEVERR_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * C::STAGE_BYTES;
          const uint32_t fb = ptx::mapa_shared(ptx::smem_u32(&full[s]), 0);
          if (lead) ptx::mbar_arrive_expect_tx(&full[s], 2u * C::STAGE_BYTES);
          if constexpr (MN) {
            // this CTA's 128 columns of A and of B: two 64-column boxes of 64 K rows each
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              ptx::tma_load_2d_pair(sa + i * C::BOX_BYTES, &tmA, fb,
                                    tc.a_row + static_cast<int>(rank) * BLOCK_M + 64 * i,
                                    kb * BLOCK_K);
              ptx::tma_load_2d_pair(sa + C::A_BYTES + i * C::BOX_BYTES, &tmB, fb,
                                    tc.b_row + static_cast<int>(rank) * (C::BN / 2) + 64 * i,
                                    kb * BLOCK_K);
            }
          } else {
            // rows past M or N are zero-filled
            ptx::tma_load_2d_pair(sa, &tmA, fb, kb * BLOCK_K,
                                  tc.a_row + static_cast<int>(rank) * BLOCK_M);
            ptx::tma_load_2d_pair(sa + C::A_BYTES, &tmB, fb, kb * BLOCK_K,
                                  tc.b_row + static_cast<int>(rank) * (C::BN / 2));
          }
        }
      }
      // rank 0's last full phases cover both CTAs' last copies: they land before the pair exits
      if (lead) {
        const uint32_t first = it > static_cast<uint32_t>(C::STAGES) ? it - C::STAGES : 0u;
        for (uint32_t j = first; j < it; ++j) {
          if (!wait_drain(&full[j % C::STAGES], (j / C::STAGES) & 1u, limit)) {
            raise_error(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && lead) {
      // ------------------------------------------------------------ MMA issuer (rank 0)
      uint32_t it = 0;
      int lt = 0;
      bool stalled = false;
      if (g.inject_stall && !ptx::mbar_wait(stall, 0u, abort_flag, limit)) {
        raise_error(g, abort_flag, DEVERR_TIMEOUT_MMA);
        stalled = true;
      }
      for (int tile = cid; !stalled && tile < total; tile += ncl, ++lt) {
        const int acc = lt & 1;
        const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
        if (!ptx::mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, limit)) {
          raise_error(g, abort_flag, DEVERR_TIMEOUT_MMA);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&full[s], ph, abort_flag, limit)) {
            raise_error(g, abort_flag, DEVERR_TIMEOUT_MMA);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < BLOCK_K / 16; ++k) {
            if constexpr (MN)  // 16 K rows = two 1024-byte atoms of each box
              ptx::umma_bf16_pair(d_tmem, ptx::smem_desc_sw128_mn(sa + k * 2048, C::BOX_BYTES),
                                  ptx::smem_desc_sw128_mn(sb + k * 2048, C::BOX_BYTES),
                                  C::IDESC_MN, (kb | k) != 0 ? 1u : 0u);
            else
              ptx::umma_bf16_pair(d_tmem, ptx::smem_desc_sw128(sa + k * 32),
                                  ptx::smem_desc_sw128(sb + k * 32), C::IDESC,
                                  (kb | k) != 0 ? 1u : 0u);
          }
          ptx::umma_commit_pair(&empty[s], 0x3);
        }
        if (!ok) break;
        ptx::umma_commit_pair(&tfull[acc], 0x3);
      }
      // all MMAs issued by this thread complete before TMEM is released
      ptx::umma_commit_pair(drain, 0x1);
      if (!wait_drain(drain, 0u, limit)) raise_error(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5, both
    // ranks): a thread owns one of this CTA's 128 output rows and walks the tile's 256 columns
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const float c = g.c, inv_c = 1.0f / g.c;
    const uint32_t tempty_lead0 = ptx::mapa_shared(ptx::smem_u32(&tempty[0]), 0);
    const uint32_t tempty_lead1 = ptx::mapa_shared(ptx::smem_u32(&tempty[1]), 0);
    int lt = 0;
    for (int tile = cid; tile < total; tile += ncl, ++lt) {
      const int acc = lt & 1;
      const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
      const TileCoord tc = decode_tile<C::BN, C::TM>(g, nt, mt, tile);
      const bool got = ptx::mbar_wait(&tfull[acc], aph, abort_flag, limit);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) raise_error(g, abort_flag, DEVERR_TIMEOUT_EPILOGUE);
        break;
      }
      ptx::tc_fence_after();
      const int row = tc.a_row + static_cast<int>(rank) * BLOCK_M + q * 32 + lane;
      const bool row_ok = row < g.M;
      // a weight gradient's output row (the row map de-interleaves gate/value rows)
      const int orow = (MN && row_ok && g.row_map) ? __ldg(g.row_map + row) : row;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * C::BN);
      if constexpr (RP) {
        // whole 32-column chunks (the launcher sets RP only for N a multiple of 256): chunk
        // ch + 1's residual is loaded before chunk ch's accumulator columns are read
        const uint4* rrow = reinterpret_cast<const uint4*>(
            g.resid + static_cast<size_t>(row_ok ? row : 0) * g.ldr + tc.n0);
        uint4 rnext[4];
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) rnext[q4] = __ldg(rrow + q4);
        }
#pragma unroll 1
        for (int ch = 0; ch < C::BN / 32; ++ch) {
          uint4 rcur[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) rcur[q4] = rnext[q4];
          if (row_ok && ch + 1 < C::BN / 32) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) rnext[q4] = __ldg(rrow + 4 * (ch + 1) + q4);
          }
          float v[32];
          ptx::tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(ch * 32), v);
          if (row_ok) store_resid_prefetched(g, row, tc.n0 + ch * 32, v, rcur);
        }
      } else {
#pragma unroll 1
        for (int ch = 0; ch < C::BN / 32; ++ch) {
          const int col0 = tc.n0 + ch * 32;
          if (col0 >= g.N) break;  // uniform across the warp
          float v[32];
          ptx::tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(ch * 32), v);
          if (row_ok) {
            if (col0 + 32 <= g.N)
              epilogue_store(g, orow, col0, v, c, inv_c);
            else
              epilogue_store_partial(g, orow, col0, g.N - col0, v);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (lead)
          ptx::mbar_arrive(&tempty[acc]);
        else
          ptx::mbar_arrive_cluster(acc == 0 ? tempty_lead0 : tempty_lead1);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer is done with this CTA's barriers, shared memory and TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

// tb: B's tensor map with BN / 2-row boxes (each CTA of a pair loads half of a tile's columns).
template <int BN, bool RP, bool MN = false>
static int launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& g,
                       cudaStream_t stream) {
  using C = GemmPairCfg<BN>;
  auto kernel = gemm_pair_kernel<BN, RP, MN>;
  if (g.ksplit > 1 || (MN ? (g.groups != 1 || g.kfull <= 0 || g.epi != EPI_F32) : g.groups > 0))
    return LMOE_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_BYTES) != cudaSuccess)
    return LMOE_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  int pairs = sms / 2;
  if (g.max_ctas > 0 && g.max_ctas / 2 < pairs) pairs = g.max_ctas / 2 > 0 ? g.max_ctas / 2 : 1;
  const int64_t tiles = ceil_div(g.M, C::TM) * ceil_div(g.N, C::BN);
  if (tiles < pairs) pairs = static_cast<int>(tiles);
  if (pairs <= 0) return LMOE_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(GEMM_THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // a persistent grid: no more pairs than can be resident at once (an SM pair shares a GPC)
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) == cudaSuccess && active > 0 &&
      active < pairs) {
    pairs = active;
    cfg.gridDim = dim3(2 * pairs);
  }
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, g) == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

template <int BN, int MT, bool RP = false>
static int launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                     const GemmArgs& g, cudaStream_t stream) {
  using C = GemmCfg<BN, MT>;
  if (cudaFuncSetAttribute(gemm_tcgen05_kernel<BN, MT, RP>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_BYTES) != cudaSuccess)
    return LMOE_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  int grid = (g.max_ctas > 0 && g.max_ctas < sms) ? g.max_ctas : sms;
  const int64_t tiles = ceil_div(g.M, BLOCK_M * MT) * ceil_div(g.N, BN) *
                        (g.groups > 0 ? g.groups : 1) * (g.ksplit > 1 ? g.ksplit : 1);
  if (tiles < grid) grid = static_cast<int>(tiles);
  if (grid <= 0) return LMOE_OK;
  return launch_pdl(gemm_tcgen05_kernel<BN, MT, RP>, grid, GEMM_THREADS, C::SMEM_BYTES, stream,
                    ta, tb, to, g) ==
                 cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_gemm(const void* A, uint64_t a_rows, int a_ld, const void* B, uint64_t b_rows,
                int b_ld, const GemmArgs& g_in, cudaStream_t stream) {
  GemmArgs g = g_in;
  g.out_tma = 0;  // set below, with the output tensor map it needs
  if (g.groups > 0 && (g.epi != EPI_F32 || !g.kseg)) return LMOE_ERR_INVALID_ARG;
  if (g.pre && ((g.epi != EPI_SITU && g.epi != EPI_SPLIT) || g.ldp % 8 ||
                (reinterpret_cast<uintptr_t>(g.pre) & 15u)))
    return LMOE_ERR_INVALID_ARG;
  if (g.groups == 0 && (g.Kd % BLOCK_K != 0 || g.Kd <= 0)) return LMOE_ERR_UNSUPPORTED;
  if (g.N <= 0) return LMOE_ERR_UNSUPPORTED;
  const bool glu = g.epi == EPI_SITU || g.epi == EPI_SPLIT;
  if (g.N % (glu ? 32 : 16) != 0 || (g.epi == EPI_SPLIT && g.split % 32 != 0))
    return LMOE_ERR_UNSUPPORTED;
  if (g.M == 0) return LMOE_OK;
  // 256-wide tiles unless N is small and not a multiple of 256 (a partial last column tile is
  // zero-filled by TMA and cut at N by the epilogue): the router's N = 896 runs as 4 column
  // tiles instead of 7, re-reading the latent half as often (61.9 -> 59.4 us at prefill)
  // N = 896 (the router over 896 experts): four whole 224-wide tiles instead of four 256-wide
  // ones, the last half empty.  A single M-tile (decode) takes 128-wide tiles: twice the column
  // tiles to spread over the SMs before the reduction is split (decode 1.181 -> 1.166 ms)
  const int bn = (g.groups == 0 && g.M > BLOCK_M && g.N % 256 != 0 && g.N > 512 &&
                  g.N % 224 == 0 && g.N <= 4 * 224)
                     ? 224
                     : (g.M <= BLOCK_M ? 128 : ((g.N % 256 == 0 || g.N > 512) ? 256 : 128));
  CUtensorMap ta, tb, to{};
  if (g.groups > 0) {
    // MN-major: a_rows / b_rows count K rows; boxes of 64 columns x 64 rows
    if (!make_tmap_bf16(&ta, A, a_rows, static_cast<uint64_t>(g.M), static_cast<uint64_t>(a_ld),
                        BLOCK_K) ||
        !make_tmap_bf16(&tb, B, b_rows, static_cast<uint64_t>(g.N), static_cast<uint64_t>(b_ld),
                        BLOCK_K))
      return LMOE_ERR_CUDA;
    // the fp32 output as (columns, rows, groups), for the epilogue's tensor stores; without
    // one (an unaligned output) the epilogue stores from its threads
    g.out_tma = GEMM_WGRAD_TMA_STORE && make_tmap_f32_out(&to, g.outf, g.N, g.M, g.groups,
                                                           g.ldf, g.group_stride)
                    ? 1
                    : 0;
  } else if (!make_tmap_bf16(&ta, A, a_rows, static_cast<uint64_t>(g.Kd),
                             static_cast<uint64_t>(a_ld), BLOCK_M) ||
             !make_tmap_bf16(&tb, B, b_rows, static_cast<uint64_t>(g.Kd),
                             static_cast<uint64_t>(b_ld), static_cast<uint32_t>(bn))) {
    return LMOE_ERR_CUDA;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  // A weight gradient over all rows of its operands (one group) with at least two 256 x 256
  // cluster tiles per SM pair: over SM pairs, like the dense tile-pair GEMMs
  if (GEMM_SM_PAIR && GEMM_WGRAD_SM_PAIR && g.groups == 1 && g.kfull > 0 && bn == 256 &&
      static_cast<uint64_t>(g.kfull) == a_rows && static_cast<uint64_t>(g.kfull) == b_rows &&
      ceil_div(g.M, 2 * BLOCK_M) * ceil_div(g.N, 256) >= 2 * static_cast<int64_t>(sms))
    return launch_pair<256, false, true>(ta, tb, g, stream);
  // Split-K when one M-tile's column tiles would leave most SMs idle (small batches): each
  // slice of K-blocks is its own tile, and a second kernel adds the slices.
  if (g.groups == 0 && g.partial && g.M <= BLOCK_M) {
    const int64_t tiles = ceil_div(g.N, bn);
    const int nkb = g.Kd / BLOCK_K;
    int64_t ks = sms / tiles;
    ks = ks < nkb / SPLITK_MIN_KB ? ks : nkb / SPLITK_MIN_KB;
    const int64_t fit = static_cast<int64_t>(g.partial_bytes /
                                             (static_cast<size_t>(g.M) * g.N * sizeof(float)));
    ks = ks < fit ? ks : fit;
    if (ks >= 2) {
      const int per = static_cast<int>(ceil_div(nkb, ks));
      GemmArgs gs = g;
      gs.ksplit = static_cast<int>(ceil_div(nkb, per));  // no slice is left empty
      const int rc = bn == 256   ? launch_bn<256, 1>(ta, tb, to, gs, stream)
                     : bn == 224 ? launch_bn<224, 1>(ta, tb, to, gs, stream)
                                 : launch_bn<128, 1>(ta, tb, to, gs, stream);
      if (rc != LMOE_OK) return rc;
      const int64_t chunks = static_cast<int64_t>(g.M) * ceil_div(g.N, 32);
      const bool warp = gs.ksplit >= SPLITK_WARP_MIN;
      const int64_t blocks = ceil_div(chunks, warp ? 8 : 256);
      const unsigned grid = static_cast<unsigned>(blocks < 16 * sms ? blocks : 16 * sms);
      if ((warp ? launch_pdl(splitk_reduce_kernel<true>, grid, 256, 0, stream, gs)
                : launch_pdl(splitk_reduce_kernel<false>, grid, 256, 0, stream, gs)) !=
          cudaSuccess)
        return LMOE_ERR_CUDA;
      if (g.extra_launches) *g.extra_launches += 1;
      return LMOE_OK;
    }
  }
  // Tile pairs (two 128-row M-tiles sharing each B stage) when the problem is dense, has at
  // least two pairs per SM and a long reduction: the pair's undivided accumulator is drained
  // while no MMA runs, which only pays when the MMAs take far longer.
  const bool pairs = g.groups == 0 && g.Kd >= GEMM_PAIR_MIN_K &&
                     ceil_div(g.M, 2 * BLOCK_M) * ceil_div(g.N, bn) >= 2 * static_cast<int64_t>(sms);
  // the output GEMM: residual epilogue over whole 256-column tiles
  const bool rp = g.epi == EPI_RESID && g.resid != nullptr && g.N % 256 == 0;
  if (GEMM_SM_PAIR && bn == 256 && pairs) {
    // over SM pairs (gemm_pair_kernel): each CTA loads 128 of a tile's 256 B rows
    CUtensorMap tbh;
    if (!make_tmap_bf16(&tbh, B, b_rows, static_cast<uint64_t>(g.Kd),
                        static_cast<uint64_t>(b_ld), 128))
      return LMOE_ERR_CUDA;
    return rp ? launch_pair<256, true>(ta, tbh, g, stream)
              : launch_pair<256, false>(ta, tbh, g, stream);
  }
  // 224-wide tiles (the router) over SM pairs once every SM pair has a tile: a single M-tile's
  // 128 x 224 tile stages 44 KB per K-block for 448 MMA cycles on its SM, a pair's half 30 KB
  if (GEMM_SM_PAIR && bn == 224 && g.Kd >= GEMM_PAIR_MIN_K &&
      ceil_div(g.M, 2 * BLOCK_M) * ceil_div(g.N, bn) >= static_cast<int64_t>(sms) / 2) {
    CUtensorMap tbh;
    if (!make_tmap_bf16(&tbh, B, b_rows, static_cast<uint64_t>(g.Kd),
                        static_cast<uint64_t>(b_ld), 112))
      return LMOE_ERR_CUDA;
    return launch_pair<224, false>(ta, tbh, g, stream);
  }
  if (bn == 256 && pairs && rp) return launch_bn<256, 2, true>(ta, tb, to, g, stream);
  if (bn == 256)
    return pairs ? launch_bn<256, 2>(ta, tb, to, g, stream)
                 : launch_bn<256, 1>(ta, tb, to, g, stream);
  if (bn == 224)
    return pairs ? launch_bn<224, 2>(ta, tb, to, g, stream)
                 : launch_bn<224, 1>(ta, tb, to, g, stream);
  return pairs ? launch_bn<128, 2>(ta, tb, to, g, stream)
               : launch_bn<128, 1>(ta, tb, to, g, stream);
}

}  // namespace lmoe
