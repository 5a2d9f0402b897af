// gemm_grouped.cu -- the routed experts' GEMMs, one small GEMM per expert segment, on the
// 5th-generation tensor cores with the operands swapped ("swap-AB"):
//
//   out[tok, r] = sum_k act[tok, k] * W[e][r, k]     for the tokens tok routed to expert e
//
// computed as D[r, tok] = W[e][r, :] . act[tok, :]^T, so that the expert's weight rows fill
// the MMA's M = 128 dimension and its tokens form N (a multiple of 32, at most TOKN).  An
// expert sees ~T*K/E tokens (146 at the K3 prefill shape, ~1 at decode): as N they cost no
// padded MMA rows, and every weight byte is staged into shared memory exactly once while
// the expert's few token rows are re-read from L2.
//
// Tiles: for each expert e, its token rows are cut into chunks of at most TOKN; each
// (expert, chunk) pair has M_w / 128 weight row-tiles, enumerated fastest so that the tiles
// sharing a token chunk run on neighbouring SMs at the same time.  The chunk counts come
// from a device-side prefix sum; nothing returns to the host.
//
// Roles as in gemm.cu: warp 0 TMA producer (one 128 x 64 weight box, a contiguous 16 KB tile
// of the packed weights, + one 32 x 64 box per 32 tokens), warp 1 TMEM owner and single-thread tcgen05.mma issuer (instruction descriptor
// with the tile's N built at run time), warps 2-5 epilogue, warps 6-9 row gatherers.  In the epilogue a thread owns
// one weight row (one output feature) and walks the tokens, so a warp writes 32 consecutive
// features of one token row per store.  Gate/value epilogue (SiTU-GLU): weight rows are
// interleaved 16 gate / 16 value, so lanes l and l+16 hold the gate and value of the same
// feature and meet through one shuffle.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace lmoe {

constexpr int GROUPED_BOX_T = 32;  // token rows per TMA box / padding granule of N

// Pipeline depth (shared-memory stages of one weight box + one token tile).  Measured at
// the K3 shapes: the gate/value GEMM (long K, gathered rows) is fastest with the deepest ring
// that fits (1.19 ms at 5 stages vs 1.28 at 4, prefill); the down GEMM (K = 512, writing the
// expert outputs) with one stage less when experts see many tokens (0.75 ms at 4 vs 0.82 at
// 5, prefill) but not at decode (~1 token per expert: 0.37 ms at 5 vs 0.39 at 4).  Single
// weight tiles now serve only the e4m3 gate/value GEMM and the one that stores its
// pre-activations, below GROUPED_PAIR_MIN_TOKENS tokens per expert (see launch_grouped_gemm).
constexpr int GROUPED_STAGES_DEEP = 5;
constexpr int GROUPED_STAGES_SHALLOW = 4;
constexpr int GROUPED_SHALLOW_MIN_TOKENS = 32;
// Weight-tile pairs: stages of two weight boxes and a token tile (56 or 64 KB): three fit,
// four (56 KB) without the epilogue's output staging.
constexpr int GROUPED_STAGES_PAIR = 3;
constexpr int GROUPED_PAIR_MIN_TOKENS = 64;  // experts' mean token count from which pairs run
// bf16 pairs over two SMs (cta_group::2, two weight tiles per SM; see grouped_gemm_pair_kernel)
// for GEMMs whose token rows are loaded by TMA
constexpr bool GROUPED_SM_PAIR = true;
constexpr bool GROUPED_OUT_TMA_STORE = true;  // the pair kernel's whole output chunks by TMA

// MW: weight row tiles per CTA tile.  MW = 2 ("weight-tile pairs") stages two 128-row
// weight tiles of the same expert with one token tile and issues two MMAs per K-step, so
// every gathered or loaded token row serves 256 output features: half the token bytes per
// FLOP, for experts with many tokens, where the token rows and not the weights bound the
// shared-memory fill.  Its accumulator pair fills TMEM (2 x 256 columns), so it is drained
// while no MMA runs (the producer keeps loading the next tile meanwhile) -- unless TOKN <= 128,
// where two pairs of 2 x 128 columns fit and the drain overlaps the next tile's MMAs.
// TOKN_: the largest token chunk the tile holds (the shared-memory token tile and the TMEM
// columns of one accumulator); the chunks themselves are set by GroupedArgs::tokn <= TOKN_.
// STAGED: the epilogue's shared-memory staging of output rows (needed by the down GEMM and by
// a gate/value GEMM that also stores its pre-activations); without it a gate/value ring of
// weight-tile pairs has room for a fourth stage.
template <int STAGES_, int MW_, int TOKN_, bool STAGED = true>
struct GroupedCfg {
  static constexpr int TOKN = TOKN_;                      // max tokens (N) per tile
  static constexpr int MW = MW_;
  static constexpr int BOX_T = GROUPED_BOX_T;             // token rows per TMA box
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K * 2;   // 16 KB per weight tile
  static constexpr int W_BYTES = MW * A_BYTES;
  static constexpr int B_BYTES = TOKN * BLOCK_K * 2;      // up to 32 KB of activations
  static constexpr int STAGE_BYTES = W_BYTES + B_BYTES;
  static constexpr int STAGES = STAGES_;
  // TMEM columns per weight tile's accumulator, and accumulator sets: two (the epilogue of
  // one tile overlaps the next tile's MMAs) unless a weight-tile pair's 2 x 256 fill TMEM
  static constexpr int ACC_COLS = (MW == 2 && TOKN <= 128) ? 128 : 256;
  static constexpr int ACC = 2 * MW * ACC_COLS <= 512 ? 2 : 1;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_OFF = STAGES * STAGE_BYTES;   // per epilogue warp 32 x 32 bf16
  static constexpr int EPI_BYTES = STAGED ? 8 * 32 * 32 * 2 : 0;
  static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  // copies of the chunk prefix sum and the expert segment offsets (E + 1 entries each) in
  // whatever shared memory is left: when both fit, the tile decode's binary search costs
  // shared-memory latency instead of 2-3 K cycles of dependent global loads per tile
  static constexpr int TAB_OFF = MISC_OFF + 16;
  static constexpr int TAB_ROOM = (232448 - 1024 - TAB_OFF) / 8;
  static constexpr int TAB_CAP = TAB_ROOM < 2048 ? TAB_ROOM : 2048;  // entries per table
  static constexpr int SMEM_BYTES = TAB_OFF + TAB_CAP * 8 + 1024;
  static_assert(TAB_CAP >= 0, "shared memory budget");
  static_assert(MW == 1 || MW == 2, "one or two weight tiles");
  static_assert(TOKN % BOX_T == 0 && TOKN % 16 == 0 && TOKN <= 256, "UMMA N range");
  static_assert(TOKN <= ACC_COLS && ACC * MW * ACC_COLS <= TMEM_COLS, "accumulators fit TMEM");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "1024-aligned tiles");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// warp 0 TMA producer, warp 1 MMA, warps 2..5 epilogue, warps 6..9 row gatherers (used when
// the activation rows are gathered through an index; otherwise a second epilogue group for
// the e4m3 down GEMM and for weight-tile pairs)
constexpr int GROUPED_EPI_WARPS = 4;
constexpr int GROUPED_GATHER_WARPS = 4;
constexpr int GROUPED_GATHER_THREADS = GROUPED_GATHER_WARPS * 32;
constexpr int GROUPED_THREADS = (2 + GROUPED_EPI_WARPS + GROUPED_GATHER_WARPS) * 32;

struct GTile {
  int e;        // expert
  int w_row;    // row coordinate of the tile's first 128 x 64 weight box (tiled layout)
  int r0;       // first weight row within the expert (output feature)
  int nw;       // weight tiles in this tile (MW, or 1 for an odd expert's last)
  int tok0;     // first token row (permuted order)
  int ntok;     // valid token rows in this tile (1..tokn)
  int npad;     // ntok rounded up to BOX_T
};

// Tile -> (expert, token chunk, weight tile group).  An expert's `count` token rows form
// ceil(count / tokn) chunks of equal size (to one row); its MW-tile groups of weight rows are
// enumerated fastest, so the tiles that share a chunk's token rows run at the same time on
// neighbouring SMs.  `ld` reads entry i of the chunk prefix sum (which = 0) or of the expert
// segment offsets (which = 1), from global memory or from a copy in shared memory.
template <int MW, typename Load>
__device__ __forceinline__ GTile decode_gtile_with(const GroupedArgs& g, int mt, int tile,
                                                   Load ld) {
  const int mg = (mt + MW - 1) / MW;  // weight tile groups per (expert, chunk)
  const int q = tile / mg;            // global (expert, chunk) index
  int lo = 0, hi = g.E;               // ct_off[lo] <= q < ct_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ld(0, mid) <= q)
      lo = mid;
    else
      hi = mid;
  }
  const int e = lo;
  const int c0 = ld(0, e);
  const int chunk = q - c0;
  const int nchunk = ld(0, e + 1) - c0;
  const int m = (tile - q * mg) * MW;
  GTile t;
  t.e = e;
  t.r0 = m * BLOCK_M;
  t.nw = min(MW, mt - m);
  t.w_row = (e * mt + m) * (g.Kd / BLOCK_K) * BLOCK_M;
  const int seg0 = ld(1, e);
  const int cnt = ld(1, e + 1) - seg0;
  // <= tokn, and every chunk non-empty; most experts have one chunk (no division)
  const int csz = nchunk == 1 ? cnt : (cnt + nchunk - 1) / nchunk;
  t.tok0 = seg0 + chunk * csz;
  t.ntok = min(csz, cnt - chunk * csz);
  t.npad = (t.ntok + GROUPED_BOX_T - 1) / GROUPED_BOX_T * GROUPED_BOX_T;
  return t;
}

template <int MW>
__device__ __forceinline__ GTile decode_gtile(const GroupedArgs& g, int mt, int tile) {
  return decode_gtile_with<MW>(g, mt, tile, [&](int which, int i) {
    return __ldg((which == 0 ? g.ct_off : g.seg_off) + i);
  });
}

__device__ __forceinline__ void graise(const GroupedArgs& g, volatile int* abort_flag,
                                       uint32_t code) {
  *abort_flag = 1;
  atomicOr(g.err, code);
}

__device__ __forceinline__ bool gwait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u && ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// SiTU-GLU, as in the dense epilogue: silu(c tanh(g/c)) * c tanh(v/c).
__device__ __forceinline__ float situ_g(float g, float v, float c, float inv_c) {
  const float gc = c * ptx::tanh_approx(g * inv_c);
  const float vc = c * ptx::tanh_approx(v * inv_c);
  return __fdividef(gc, 1.0f + __expf(fminf(-gc, 80.0f))) * vc;
}

// tanh to ~2^-20 relative: below |x| = 1/4 its odd Taylor polynomial through x^9 (the next
// term, 1382/155925 x^11, is < 1.5e-8 of tanh there), above it (1 - e) / (1 + e) with
// e = exp(-2|x|), where the subtraction loses no significant bits.
// Both branches are evaluated and one is selected: a warp vote to skip the exponential
// measured slower (it serialises the unrolled epilogue loop).
__device__ __forceinline__ float tanh_close(float x) {
  const float ax = fabsf(x);
  const float x2 = x * x;
  float p = fmaf(x2, 62.0f / 2835.0f, -17.0f / 315.0f);
  p = fmaf(x2, p, 2.0f / 15.0f);
  p = fmaf(x2, p, -1.0f / 3.0f);
  p = fmaf(x2 * x, p, x);
  const float e = __expf(-2.0f * ax);
  const float t = copysignf(__fdividef(1.0f - e, 1.0f + e), x);
  return ax < 0.25f ? p : t;
}

// SiTU-GLU for the FP8 path, which quantises h next: an e4m3 code moves when its input
// moves by 2^-4 relative, so h must carry little more error than the fp32 GEMM sums
// themselves (the MUFU tanh approximation, ~2^-11, would move ~1 % of the codes).
__device__ __forceinline__ float situ_close(float g, float v, float c, float inv_c) {
  const float gc = c * tanh_close(g * inv_c);
  const float vc = c * tanh_close(v * inv_c);
  return __fdividef(gc, 1.0f + __expf(fminf(-gc, 80.0f))) * vc;
}

template <int STAGES_, bool FP8, int MW, int TOKN_, bool STAGED>
__global__ void __launch_bounds__(GROUPED_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmX, const GroupedArgs g) {
  using C = GroupedCfg<STAGES_, MW, TOKN_, STAGED>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  __nv_bfloat16* epi_stage = reinterpret_cast<__nv_bfloat16*>(smem + C::EPI_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (g.M_w + BLOCK_M - 1) / BLOCK_M;
  const int nk = g.Kd / BLOCK_K;
  const uint64_t limit = g.timeout_ns;

  if (threadIdx.x == 0) {
    // a stage is full once the TMA bytes have landed and, when rows are gathered, every
    // gathering thread's copies have landed too
    const uint32_t full_count = 1u + (g.gather ? GROUPED_GATHER_THREADS : 0u);
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(&full[s], full_count);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      // with nothing gathered (the down GEMM), warps 6..9 join the epilogue for e4m3
      // operands and for weight-tile pairs
      ptx::mbar_init(&tempty[a], (((FP8 || MW == 2) && !g.gather) ? 2 * GROUPED_EPI_WARPS
                                                                 : GROUPED_EPI_WARPS) * 32);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // from here on: the previous kernel's outputs (segments, rows) are visible
  pdl_launch_dependents();
  int32_t* tab = reinterpret_cast<int32_t*>(smem + C::TAB_OFF);
  const bool tab_smem = g.E < C::TAB_CAP;  // both tables' E + 1 entries fit
  if (tab_smem) {
    for (int i = threadIdx.x; i <= g.E; i += blockDim.x) {
      tab[i] = __ldg(g.ct_off + i);
      tab[C::TAB_CAP + i] = __ldg(g.seg_off + i);
    }
    __syncthreads();
  }
  auto decode = [&](int tile) {
    return decode_gtile_with<MW>(g, mt, tile, [&](int which, int i) {
      return tab_smem ? tab[which * C::TAB_CAP + i]
                      : __ldg((which == 0 ? g.ct_off : g.seg_off) + i);
    });
  };
  const int total = (tab_smem ? tab[g.E] : __ldg(g.ct_off + g.E)) * ((mt + MW - 1) / MW);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      const uint64_t w_policy = ptx::l2_policy_evict_first();  // for weights read once
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const GTile t = decode(tile);
        const int nbox = g.gather ? 0 : t.npad / C::BOX_T;
        const uint32_t bytes = static_cast<uint32_t>(t.nw) * C::A_BYTES +
                               static_cast<uint32_t>(nbox) * C::BOX_T * BLOCK_K * 2;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, limit)) {
            graise(g, abort_flag, DEVERR_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * C::STAGE_BYTES;
          uint8_t* sb = sa + C::W_BYTES;
          ptx::mbar_arrive_expect_tx(&full[s], bytes);
          if constexpr (MW == 1) {
            if (g.evict_first)
              ptx::tma_load_2d_hint(sa, &tmW, &full[s], 0, t.w_row + kb * BLOCK_M, w_policy);
            else
              ptx::tma_load_2d(sa, &tmW, &full[s], 0, t.w_row + kb * BLOCK_M);
          } else {
            for (int w = 0; w < t.nw; ++w) {  // an expert's row tiles are nk boxes apart
              const int wr = t.w_row + (w * nk + kb) * BLOCK_M;
              if (g.evict_first)
                ptx::tma_load_2d_hint(sa + w * C::A_BYTES, &tmW, &full[s], 0, wr, w_policy);
              else
                ptx::tma_load_2d(sa + w * C::A_BYTES, &tmW, &full[s], 0, wr);
            }
          }
          for (int b = 0; b < nbox; ++b)
            ptx::tma_load_2d(sb + b * C::BOX_T * BLOCK_K * 2, &tmX, &full[s], kb * BLOCK_K,
                             t.tok0 + b * C::BOX_T);
        }
      }
      // every issued copy must land before the CTA may exit
      const uint32_t first = it > static_cast<uint32_t>(C::STAGES) ? it - C::STAGES : 0u;
      for (uint32_t j = first; j < it; ++j) {
        if (!gwait_drain(&full[j % C::STAGES], (j / C::STAGES) & 1u, limit)) {
          graise(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
          break;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      uint32_t it = 0;
      int lt = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++lt) {
        const GTile t = decode(tile);
        const uint32_t idesc = FP8 ? ptx::idesc_e4m3_f32(BLOCK_M, t.npad)
                                   : ptx::idesc_bf16_f32(BLOCK_M, t.npad);
        const int acc = C::ACC == 2 ? (lt & 1) : 0;
        const uint32_t aph = C::ACC == 2 ? (static_cast<uint32_t>(lt >> 1) & 1u)
                                         : (static_cast<uint32_t>(lt) & 1u);
        if (!ptx::mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, limit)) {
          graise(g, abort_flag, DEVERR_TIMEOUT_MMA);
          break;
        }
        ptx::tc_fence_after();
        // weight tile w of the tile accumulates at TMEM columns (acc * MW + w) * ACC_COLS
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MW * C::ACC_COLS);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&full[s], ph, abort_flag, limit)) {
            graise(g, abort_flag, DEVERR_TIMEOUT_MMA);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          if (g.gather) ptx::fence_proxy_async_smem();  // rows written by cp.async
          const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + C::W_BYTES;
#pragma unroll
          for (int k = 0; k < BLOCK_K / 16; ++k) {  // 32 bytes of K per instruction
#pragma unroll
            for (int w = 0; w < MW; ++w) {
              if (MW > 1 && w >= t.nw) break;
              const uint32_t dw = d_tmem + static_cast<uint32_t>(w * C::ACC_COLS);
              const uint32_t aw = sa + w * C::A_BYTES + k * 32;
              if constexpr (FP8)
                ptx::umma_e4m3(dw, ptx::smem_desc_sw128(aw), ptx::smem_desc_sw128(sb + k * 32),
                               idesc, (kb | k) != 0 ? 1u : 0u);
              else
                ptx::umma_bf16(dw, ptx::smem_desc_sw128(aw), ptx::smem_desc_sw128(sb + k * 32),
                               idesc, (kb | k) != 0 ? 1u : 0u);
            }
          }
          ptx::umma_commit(&empty[s]);
        }
        if (!ok) break;
        ptx::umma_commit(&tfull[acc]);
      }
      ptx::umma_commit(drain);
      if (!gwait_drain(drain, 0u, limit)) graise(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp >= 2 + GROUPED_EPI_WARPS && (g.gather || (!FP8 && MW == 1))) {
    // ------------------------------------------------------------ row gatherers (warps 6..9)
    // Thread gt copies 16-byte chunk (gt & 7) of rows gt/8 + 16 j of each stage's token
    // tile, from the activation row src = gather[permuted row], into the 128-byte-swizzled
    // K-major layout the MMA reads; its arrival on the stage's barrier fires when they land.
    if (g.gather) {
      const int gt = threadIdx.x - (2 + GROUPED_EPI_WARPS) * 32;
      const int chunk = gt & 7;
      constexpr int J = C::TOKN / 16;  // rows per thread
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const GTile t = decode(tile);
        const __nv_bfloat16* src[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int row = (gt >> 3) + 16 * j;
          const int tok = t.tok0 + (row < t.ntok ? row : t.ntok - 1);  // pad: a valid row
          src[j] = g.x + static_cast<size_t>(__ldg(g.gather + tok)) * g.ldx + chunk * 8;
        }
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, limit)) {
            graise(g, abort_flag, DEVERR_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          const uint32_t sb = ptx::smem_u32(smem + s * C::STAGE_BYTES + C::W_BYTES);
#pragma unroll
          for (int j = 0; j < J; ++j) {
            const int row = (gt >> 3) + 16 * j;
            if (row < t.npad)
              ptx::cp_async_16(sb + row * 128 + ((chunk ^ (row & 7)) << 4), src[j] + kb * BLOCK_K);
          }
          ptx::cp_async_mbar_arrive_noinc(&full[s]);
        }
      }
      ptx::cp_async_wait_all();
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5; with
    // nothing gathered, also 6..9: for the e4m3 down GEMM the two groups take the even and
    // odd token chunks -- its mainloop is half as long as the bf16 one, so the output stores
    // bound it -- and for weight-tile pairs one weight tile each).  The bf16 down GEMM of
    // single weight tiles measured slower with the second group (its warps only poll).
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const bool two = (FP8 || MW == 2) && !g.gather;
    const int eg = (warp - 2) / GROUPED_EPI_WARPS;
    const int ch0 = (two && MW == 1) ? eg : 0, chstep = (two && MW == 1) ? 2 : 1;
    const int w0 = (two && MW == 2) ? eg : 0, wstep = (two && MW == 2) ? 2 : 1;
    const float c = g.c, inv_c = 1.0f / g.c;
    int lt = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++lt) {
      const int acc = C::ACC == 2 ? (lt & 1) : 0;
      const uint32_t aph = C::ACC == 2 ? (static_cast<uint32_t>(lt >> 1) & 1u)
                                       : (static_cast<uint32_t>(lt) & 1u);
      // the tile and, with fp8, its scales are fetched before the accumulator is ready, so
      // their load latency hides under the tile's MMAs
      const GTile t = decode(tile);
      constexpr int NCH = C::TOKN / 32;    // token chunks of a tile
      float w_s[MW];                       // this thread's weight row scale, per weight tile
      float x_s[NCH];                      // lane l: scale of token 32 c + l of the tile
#pragma unroll
      for (int w = 0; w < MW; ++w) w_s[w] = 1.0f;
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) x_s[cc] = 0.0f;
      if constexpr (FP8) {
#pragma unroll
        for (int w = 0; w < MW; ++w)  // rows past the expert's last tile: a finite dummy
          w_s[w] = w < t.nw ? __ldg(g.w_scale + static_cast<size_t>(t.e) * mt * BLOCK_M + t.r0 +
                                    w * BLOCK_M + q * 32 + lane)
                            : 0.0f;
        int src[NCH];
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          const int p = t.tok0 + cc * 32 + lane;
          src[cc] = (cc * 32 + lane < t.ntok) ? (g.gather ? __ldg(g.gather + p) : p) : -1;
        }
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc)
          x_s[cc] = src[cc] >= 0 ? __ldg(g.x_scale + src[cc]) : 0.0f;
      }
      const bool got = ptx::mbar_wait(&tfull[acc], aph, abort_flag, limit);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) graise(g, abort_flag, DEVERR_TIMEOUT_EPILOGUE);
        break;
      }
      ptx::tc_fence_after();
#pragma unroll 1
      for (int w = w0; w < (MW == 1 ? 1 : t.nw); w += wstep) {
        const int r0w = t.r0 + w * BLOCK_M;    // first weight row of weight tile w
        const int r = r0w + q * 32 + lane;     // weight row of this thread within the expert
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>((acc * MW + w) * C::ACC_COLS);
        const bool row_ok = r < g.M_w;  // the last weight tile of an expert may be partial
#pragma unroll 1
        for (int ch = ch0; ch * 32 < t.npad; ch += chstep) {
          const int nv = min(32, t.ntok - ch * 32);
          // The e4m3 down GEMM (weight-tile pairs, bf16 outputs; row_ok is warp-uniform: M_w
          // is a multiple of 64): the warp's 32 rows x 32 tokens into its staging slot as token
          // rows, per 16 TMEM lanes as 8 x 8 blocks in fragment layout stored transposed
          // (stmatrix); the slot's 16-byte pieces are XOR-swizzled by (token / 2) % 4.  Only
          // these instantiations carry it: compiled into the e4m3 gate/value GEMM it slowed
          // that GEMM's SiTU epilogue (0.644 -> 0.785 ms at prefill) without running.
          if constexpr (FP8 && MW == 2 && STAGED) {
            if (g.epi != EPI_SITU) {
              if (!row_ok) continue;
              __nv_bfloat16* st = epi_stage + (warp - 2) * (32 * 32);
              float xs = x_s[0], ws = w_s[0];  // lane l's token scale and row scale
#pragma unroll
              for (int cc = 1; cc < NCH; ++cc) xs = ch == cc ? x_s[cc] : xs;
#pragma unroll
              for (int ww = 1; ww < MW; ++ww) ws = w == ww ? w_s[ww] : ws;
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                float f[16];
                ptx::tmem_ld_16x256b_x4(tbase + (static_cast<uint32_t>(16 * hf) << 16) +
                                            static_cast<uint32_t>(ch * 32),
                                        f);
                // e4m3 scales as v * ws * xs below, per (row, token) of the fragment
                const float wa = __shfl_sync(0xffffffffu, ws, 16 * hf + (lane >> 2));
                const float wb = __shfl_sync(0xffffffffu, ws, 16 * hf + 8 + (lane >> 2));
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                  const float xa = __shfl_sync(0xffffffffu, xs, 8 * n + 2 * (lane & 3));
                  const float xb = __shfl_sync(0xffffffffu, xs, 8 * n + 2 * (lane & 3) + 1);
                  f[4 * n] = f[4 * n] * wa * xa;
                  f[4 * n + 1] = f[4 * n + 1] * wa * xb;
                  f[4 * n + 2] = f[4 * n + 2] * wb * xa;
                  f[4 * n + 3] = f[4 * n + 3] * wb * xb;
                }
                uint32_t m[8];
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                  const __nv_bfloat162 a = __floats2bfloat162_rn(f[4 * n], f[4 * n + 1]);
                  const __nv_bfloat162 b = __floats2bfloat162_rn(f[4 * n + 2], f[4 * n + 3]);
                  m[2 * n] = *reinterpret_cast<const uint32_t*>(&a);
                  m[2 * n + 1] = *reinterpret_cast<const uint32_t*>(&b);
                }
#pragma unroll
                for (int call = 0; call < 2; ++call) {
                  const int i = lane >> 3;
                  const int tok = 8 * (2 * call + (i >> 1)) + (lane & 7);
                  const int pc = (2 * hf + (i & 1)) ^ ((tok >> 1) & 3);
                  ptx::stmatrix_x4_trans(ptx::smem_u32(st + tok * 32 + pc * 8), m[4 * call],
                                         m[4 * call + 1], m[4 * call + 2], m[4 * call + 3]);
                }
              }
              __syncwarp();
              const int piece = lane & 3;
#pragma unroll
              for (int j0 = 0; j0 < 32; j0 += 8) {
                const int j = j0 + (lane >> 2);
                const uint4 val =
                    *reinterpret_cast<const uint4*>(st + j * 32 + (piece ^ ((j >> 1) & 3)) * 8);
                if (j < nv)
                  *reinterpret_cast<uint4*>(g.out +
                                            static_cast<size_t>(t.tok0 + ch * 32 + j) * g.ldo +
                                            r0w + q * 32 + piece * 8) = val;
              }
              __syncwarp();
              continue;
            }
          }
          float v[32];
          ptx::tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(ch * 32), v);
          if constexpr (FP8) {
            float xs = x_s[0];  // this chunk's scales (a register select, no local memory)
#pragma unroll
            for (int cc = 1; cc < NCH; ++cc) xs = ch == cc ? x_s[cc] : xs;
            float ws = w_s[0];
#pragma unroll
            for (int ww = 1; ww < MW; ++ww) ws = w == ww ? w_s[ww] : ws;
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = v[j] * ws * __shfl_sync(0xffffffffu, xs, j);
          }
          __nv_bfloat16* orow = g.out + static_cast<size_t>(t.tok0 + ch * 32) * g.ldo;
          // through shared memory: the warp's 32 rows x 32 tokens become, per token, four
          // 16-byte pieces of its output row, so a store instruction writes 8 tokens' rows
          // instead of one
          auto staged_store = [&](__nv_bfloat16* base, int ld) {
            if constexpr (!STAGED) return;  // the launcher pairs these epilogues with staging
            __nv_bfloat16* st = epi_stage + (warp - 2) * (32 * 32);
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j * 32 + lane] = __float2bfloat16_rn(v[j]);
            __syncwarp();
            const int piece = lane & 3;
#pragma unroll
            for (int j0 = 0; j0 < 32; j0 += 8) {
              const int j = j0 + (lane >> 2);
              const uint4 val = *reinterpret_cast<const uint4*>(st + j * 32 + piece * 8);
              if (j < nv)
                *reinterpret_cast<uint4*>(base + static_cast<size_t>(t.tok0 + ch * 32 + j) * ld +
                                          r0w + q * 32 + piece * 8) = val;
            }
            __syncwarp();
          };
          if (g.epi == EPI_SITU) {
            if (g.pre) staged_store(g.pre, g.ldp);  // the pre-activations, for a backward pass
            // rows r (gate, lanes 0..15) and r + 16 (value, lanes 16..31) of one 32-row group
            // hold feature f; lanes 0..15 evaluate it for the even tokens, lanes 16..31 for
            // the odd ones, so every SiTU evaluation uses the whole warp
            const int f = ((r0w + q * 32) >> 1) + (lane & 15);
            const bool hi = lane >= 16;
#pragma unroll
            for (int jp = 0; jp < 16; ++jp) {
              const float x0 = __shfl_xor_sync(0xffffffffu, v[2 * jp], 16);
              const float x1 = __shfl_xor_sync(0xffffffffu, v[2 * jp + 1], 16);
              const float gv = hi ? x1 : v[2 * jp];       // gate of token 2jp (+1 on hi lanes)
              const float vv = hi ? v[2 * jp + 1] : x0;   // value of the same token
              const int j = 2 * jp + (hi ? 1 : 0);
              // padding tokens hold finite values (a repeated valid row, or a zero scale)
              const float hv = FP8 ? situ_close(gv, vv, c, inv_c) : situ_g(gv, vv, c, inv_c);
              if (j < nv) orow[static_cast<size_t>(j) * g.ldo + f] = __float2bfloat16_rn(hv);
            }
          } else if (row_ok) {
            staged_store(g.out, g.ldo);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[acc]);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------
// Weight tiles over an SM pair (tcgen05 cta_group::2), for the GEMMs whose token rows are
// loaded by TMA (the routed down GEMM, the backward's grouped GEMMs).
//
// A cluster of two CTAs on two SMs computes one (expert, token chunk, 512 weight rows) tile
// with MMAs of M = 256: rank r holds weight tiles 2r and 2r + 1 (128 rows each) of the group
// and the r-th half of the chunk's padded token rows (npad / 2, a multiple of 16).  Rank 0
// issues the MMAs; each reads both CTAs' shared memory at the same offsets, and each CTA's
// TMEM receives its 256 weight rows x all npad tokens.  Per K-block an SM stages 32 KB of
// weights and at most 16 KB of token rows for 256 x npad x 64 of the MMA, against 32 KB +
// 32 KB for the same share as a weight-tile pair on one SM.  The two accumulators take all
// 512 TMEM columns and are drained while no MMA runs, as on one SM.  (With one weight tile per
// CTA, two accumulator sets fit and the drain overlaps the next tile's MMAs; that measured
// slower.  The gate/value GEMM, whose rows are gathered, stays on one SM: a gathered variant
// with a forwarding thread for the peer's rows was slower there.)
//
// Synchronisation (every wait bounded):
// - full[s] of rank 0 completes when both CTAs' TMA bytes for stage s have landed: rank 0's
//   producer expects both CTAs' bytes, rank 1's copies complete on rank 0's barrier.
// - empty[s] and tfull of both CTAs get one arrival each from rank 0's commits (multicast).
// - tempty of rank 0 gets one arrival per epilogue warp of both CTAs (remote ones with the
//   default arrive semantics: a release at cluster scope made each take ~1 us).
// - a cluster barrier after the barriers are initialised, and one before TMEM is freed and the
//   CTAs exit, so that neither CTA leaves while its peer may still signal its barriers or read
//   its shared memory.
template <int STAGES_, int TOKN_>
struct GroupedPairCfg {
  static constexpr int MW = 2;                           // weight tiles per CTA
  static constexpr int TOKN = TOKN_;                     // max tokens (N) per cluster tile
  static constexpr int HALF = TOKN / 2;                  // token rows per CTA
  static constexpr int BOX_T = 16;                       // token rows per TMA box
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K * 2;  // 16 KB
  static constexpr int W_BYTES = MW * A_BYTES;
  static constexpr int B_BYTES = HALF * BLOCK_K * 2;     // up to 16 KB
  static constexpr int STAGE_BYTES = W_BYTES + B_BYTES;
  static constexpr int STAGES = STAGES_;
  static constexpr int ACC_COLS = 256;                   // TMEM columns per weight tile
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 8;                    // warps 2..9
  static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr int EPI_BYTES = EPI_WARPS * 32 * 32 * 2;  // a 2 KB staging slot per warp
  static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 3;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  // copies of the chunk prefix sum and the expert segment offsets (E + 1 entries each) in the
  // rest of the shared memory: the tile decode's binary search then costs shared-memory
  // latency instead of 2-3 K cycles of dependent global loads per tile
  static constexpr int TAB_OFF = MISC_OFF + 16;
  static constexpr int TAB_ROOM = (232448 - 1024 - TAB_OFF) / 8;
  static constexpr int TAB_CAP = TAB_ROOM < 2048 ? TAB_ROOM : 2048;  // entries per table
  static constexpr int SMEM_BYTES = TAB_OFF + TAB_CAP * 8 + 1024;
  static_assert(TOKN % 32 == 0 && TOKN <= ACC_COLS && MW * ACC_COLS <= TMEM_COLS,
                "UMMA N range; the accumulators fit TMEM");
  static_assert(TAB_CAP >= 1024, "room for the decode tables of up to 1023 experts");
  static_assert(B_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "1024-aligned tiles");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// tmO (used when g.out_tma): the output as 32 x 32 boxes with the 64-byte swizzle, the layout of
// an epilogue warp's staging slot.
template <int STAGES_, int TOKN_>
__global__ void __launch_bounds__(GROUPED_THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmO, const GroupedArgs g) {
  using C = GroupedPairCfg<STAGES_, TOKN_>;
  constexpr int MW = C::MW;
  constexpr int CW = 2 * MW;  // weight tiles per cluster tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  __nv_bfloat16* epi_stage = reinterpret_cast<__nv_bfloat16*>(smem + C::EPI_OFF);

  const uint32_t rank = ptx::cluster_ctarank();  // rank 0 issues the MMAs
  const bool lead = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = g.M_w / BLOCK_M;  // a multiple of CW: the launcher checks
  const int nk = g.Kd / BLOCK_K;
  const uint64_t limit = g.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);  // rank 0's producer; the bytes come from both CTAs
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::mbar_init(tempty, 2 * C::EPI_WARPS);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
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
  pdl_wait();
  pdl_launch_dependents();
  int32_t* tab = reinterpret_cast<int32_t*>(smem + C::TAB_OFF);
  const bool tab_smem = g.E < C::TAB_CAP;  // both tables' E + 1 entries fit
  if (tab_smem) {
    for (int i = threadIdx.x; i <= g.E; i += blockDim.x) {
      tab[i] = __ldg(g.ct_off + i);
      tab[C::TAB_CAP + i] = __ldg(g.seg_off + i);
    }
    __syncthreads();
  }
  auto decode = [&](int tile) {
    return decode_gtile_with<CW>(g, mt, tile, [&](int which, int i) {
      return tab_smem ? tab[which * C::TAB_CAP + i]
                      : __ldg((which == 0 ? g.ct_off : g.seg_off) + i);
    });
  };
  const int total = (tab_smem ? tab[g.E] : __ldg(g.ct_off + g.E)) * (mt / CW);
  const int cid = static_cast<int>(ptx::cluster_id_x());
  const int ncl = static_cast<int>(ptx::ncluster_x());

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both ranks)
      const uint64_t w_policy = ptx::l2_policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl) {
        const GTile t = decode(tile);
        const int half = t.npad / 2;
        const int nbox = half / C::BOX_T;
        const uint32_t bytes =  // both CTAs' copies: rank 0 expects them all
            2u * (static_cast<uint32_t>(C::W_BYTES) +
                  static_cast<uint32_t>(nbox) * C::BOX_T * BLOCK_K * 2u);
        // this CTA's weight tiles are rank * MW .. rank * MW + MW - 1 of the cluster tile's;
        // an expert's row tiles are nk boxes apart
        const int wr0 = t.w_row + static_cast<int>(rank) * MW * nk * BLOCK_M;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, limit)) {
            graise(g, abort_flag, DEVERR_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * C::STAGE_BYTES;
          uint8_t* sb = sa + C::W_BYTES;
          const uint32_t fb = ptx::mapa_shared(ptx::smem_u32(&full[s]), 0);
          if (lead) ptx::mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
          for (int w = 0; w < MW; ++w) {
            const int wr = wr0 + (w * nk + kb) * BLOCK_M;
            if (g.evict_first)
              ptx::tma_load_2d_pair_hint(sa + w * C::A_BYTES, &tmW, fb, 0, wr, w_policy);
            else
              ptx::tma_load_2d_pair(sa + w * C::A_BYTES, &tmW, fb, 0, wr);
          }
          for (int b = 0; b < nbox; ++b)
            ptx::tma_load_2d_pair(sb + b * C::BOX_T * BLOCK_K * 2, &tmX, fb, kb * BLOCK_K,
                                  t.tok0 + static_cast<int>(rank) * half + b * C::BOX_T);
        }
      }
      // rank 0's last full phases cover both CTAs' last copies: they land before the pair exits
      if (lead) {
        const uint32_t first = it > static_cast<uint32_t>(C::STAGES) ? it - C::STAGES : 0u;
        for (uint32_t j = first; j < it; ++j) {
          if (!ptx::mbar_wait(&full[j % C::STAGES], (j / C::STAGES) & 1u, abort_flag, limit)) {
            graise(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
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
      for (int tile = cid; tile < total; tile += ncl, ++lt) {
        const GTile t = decode(tile);
        const uint32_t idesc = ptx::idesc_bf16_f32(2 * BLOCK_M, t.npad);
        if (!ptx::mbar_wait(tempty, (static_cast<uint32_t>(lt) & 1u) ^ 1u, abort_flag, limit)) {
          graise(g, abort_flag, DEVERR_TIMEOUT_MMA);
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % C::STAGES);
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!ptx::mbar_wait(&full[s], ph, abort_flag, limit)) {
            graise(g, abort_flag, DEVERR_TIMEOUT_MMA);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + C::W_BYTES;
#pragma unroll
          for (int k = 0; k < BLOCK_K / 16; ++k) {  // 32 bytes of K per instruction
#pragma unroll
            for (int w = 0; w < MW; ++w)  // weight tile w accumulates at TMEM column w * 256
              ptx::umma_bf16_pair(tmem_base + static_cast<uint32_t>(w * C::ACC_COLS),
                                  ptx::smem_desc_sw128(sa + w * C::A_BYTES + k * 32),
                                  ptx::smem_desc_sw128(sb + k * 32), idesc,
                                  (kb | k) != 0 ? 1u : 0u);
          }
          ptx::umma_commit_pair(&empty[s], 0x3);
        }
        if (!ok) break;
        ptx::umma_commit_pair(tfull, 0x3);
      }
      ptx::umma_commit_pair(drain, 0x1);
      if (!ptx::mbar_wait(drain, 0u, abort_flag, limit))
        graise(g, abort_flag, DEVERR_TIMEOUT_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both ranks)
    // warps 2..9; the two groups of four take the even and odd 32-token chunks.  A thread owns
    // one weight row of each of this CTA's two tiles (TMEM lane quarter warp & 3) and writes it
    // for the tokens of both halves, through a per-warp staging slot as 16-byte pieces of the
    // token rows.
    const int q = warp & 3;
    const int eg = (warp - 2) / GROUPED_EPI_WARPS;
    const uint32_t tempty_lead = ptx::mapa_shared(ptx::smem_u32(tempty), 0);
    __nv_bfloat16* st = epi_stage + (warp - 2) * (32 * 32);
    bool pending = false;  // a tensor store of the slot may still be reading it
    int lt = 0;
    for (int tile = cid; tile < total; tile += ncl, ++lt) {
      const GTile t = decode(tile);  // before the wait: its loads hide there
      const bool got = ptx::mbar_wait(tfull, static_cast<uint32_t>(lt) & 1u, abort_flag, limit);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) graise(g, abort_flag, DEVERR_TIMEOUT_EPILOGUE);
        break;
      }
      ptx::tc_fence_after();
#pragma unroll 1
      for (int w = 0; w < MW; ++w) {
        // this CTA's weight tile w: its first weight row within the expert
        const int r0w = t.r0 + (static_cast<int>(rank) * MW + w) * BLOCK_M;
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(w * C::ACC_COLS);
#pragma unroll 1
        for (int ch = eg; ch * 32 < t.npad; ch += 2) {
          const int nv = min(32, t.ntok - ch * 32);
          if (pending) {  // the slot's last tensor store has read it
            if (lane == 0) ptx::bulk_wait_group_read<0>();
            __syncwarp();
            pending = false;
          }
          // the warp's 32 weight rows x 32 tokens into the staging slot as [token][row] bf16,
          // token rows of 64 bytes whose 16-byte pieces are XOR-swizzled by (token / 2) % 4:
          // per 16 TMEM lanes, 8 x 8 blocks in fragment layout stored transposed (stmatrix)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            float f[16];
            ptx::tmem_ld_16x256b_x4(
                tbase + (static_cast<uint32_t>(16 * hf) << 16) + static_cast<uint32_t>(ch * 32), f);
            uint32_t m[8];  // m[2n]: rows 16hf + 0..7, m[2n + 1]: rows 16hf + 8..15; tokens 8n..
#pragma unroll
            for (int n = 0; n < 4; ++n) {
              const __nv_bfloat162 a = __floats2bfloat162_rn(f[4 * n], f[4 * n + 1]);
              const __nv_bfloat162 b = __floats2bfloat162_rn(f[4 * n + 2], f[4 * n + 3]);
              m[2 * n] = *reinterpret_cast<const uint32_t*>(&a);
              m[2 * n + 1] = *reinterpret_cast<const uint32_t*>(&b);
            }
#pragma unroll
            for (int call = 0; call < 2; ++call) {
              const int i = lane >> 3;  // the matrix whose row this thread addresses
              const int tok = 8 * (2 * call + (i >> 1)) + (lane & 7);
              const int pc = (2 * hf + (i & 1)) ^ ((tok >> 1) & 3);
              ptx::stmatrix_x4_trans(ptx::smem_u32(st + tok * 32 + pc * 8), m[4 * call],
                                     m[4 * call + 1], m[4 * call + 2], m[4 * call + 3]);
            }
          }
          if (g.out_tma && nv == 32) {
            // a whole chunk: one tensor store of the slot (32 rows of this warp x 32 tokens)
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(&tmO, st, r0w + q * 32, t.tok0 + ch * 32);
              ptx::bulk_commit_group();
            }
            pending = true;
            continue;
          }
          __syncwarp();
          const int piece = lane & 3;
#pragma unroll
          for (int j0 = 0; j0 < 32; j0 += 8) {
            const int j = j0 + (lane >> 2);
            const uint4 val =
                *reinterpret_cast<const uint4*>(st + j * 32 + (piece ^ ((j >> 1) & 3)) * 8);
            if (j < nv)
              *reinterpret_cast<uint4*>(g.out + static_cast<size_t>(t.tok0 + ch * 32 + j) * g.ldo +
                                        r0w + q * 32 + piece * 8) = val;
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (lead)
          ptx::mbar_arrive(tempty);
        else
          ptx::mbar_arrive_cluster(tempty_lead);
      }
    }
    // the tensor stores complete before the CTA leaves (they read its shared memory)
    if (lane == 0) ptx::bulk_wait_group_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer is done with this CTA's barriers, shared memory and TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <int STAGES_, int TOKN_>
static int launch_grouped_pair(const CUtensorMap& tw, const CUtensorMap& tx, uint64_t x_rows,
                               const GroupedArgs& g_in, cudaStream_t stream) {
  // the output for tensor stores of whole 32-token chunks: it has the token operand's rows
  GroupedArgs g = g_in;
  CUtensorMap to{};
  g.out_tma = GROUPED_OUT_TMA_STORE && make_tmap_bf16_out32(&to, g.out, x_rows, g.M_w, g.ldo);
  using C = GroupedPairCfg<STAGES_, TOKN_>;
  auto kernel = grouped_gemm_pair_kernel<STAGES_, TOKN_>;
  if (g.tokn > TOKN_) return LMOE_ERR_UNSUPPORTED;
  if (g.gather || g.epi != EPI_BF16 || g.fp8 || g.M_w % (2 * C::MW * BLOCK_M) != 0)
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(GROUPED_THREADS);
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
  return cudaLaunchKernelEx(&cfg, kernel, tw, tx, to, g) == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

template <int STAGES_, bool FP8, int MW, int TOKN_, bool STAGED = true>
static int launch_grouped_stages(const CUtensorMap& tw, const CUtensorMap& tx,
                                 const GroupedArgs& g, cudaStream_t stream) {
  using C = GroupedCfg<STAGES_, MW, TOKN_, STAGED>;
  auto kernel = grouped_gemm_kernel<STAGES_, FP8, MW, TOKN_, STAGED>;
  if (g.tokn > TOKN_) return LMOE_ERR_UNSUPPORTED;
  if (!STAGED && (g.epi != EPI_SITU || g.pre)) return LMOE_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_BYTES) != cudaSuccess)
    return LMOE_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  const int grid = (g.max_ctas > 0 && g.max_ctas < sms) ? g.max_ctas : sms;
  return launch_pdl(kernel, grid, GROUPED_THREADS, C::SMEM_BYTES, stream, tw, tx, g) ==
                 cudaSuccess
             ? LMOE_OK
             : LMOE_ERR_CUDA;
}

int launch_grouped_gemm(const void* W, const void* X, uint64_t x_rows, int x_ld,
                        const GroupedArgs& g, cudaStream_t stream) {
  const int kgran = g.fp8 ? 2 * BLOCK_K : BLOCK_K;  // elements per 128-byte K-block
  if (g.M_w <= 0 || g.Kd % kgran != 0 || g.Kd <= 0 || x_rows == 0) return LMOE_ERR_UNSUPPORTED;
  if (g.epi != EPI_SITU && g.epi != EPI_BF16) return LMOE_ERR_UNSUPPORTED;
  if (g.epi == EPI_SITU && g.M_w % BLOCK_M != 0) return LMOE_ERR_UNSUPPORTED;
  if (g.tokn != GROUPED_TOKN && g.tokn != GROUPED_TOKN_WIDE && g.tokn != GROUPED_TOKN_NARROW)
    return LMOE_ERR_INVALID_ARG;
  if (g.fp8 && (!g.w_scale || !g.x_scale || x_ld % 2 != 0)) return LMOE_ERR_INVALID_ARG;
  if (g.pre && (g.epi != EPI_SITU || g.ldp % 8 != 0 || g.ldp < g.M_w ||
                (reinterpret_cast<uintptr_t>(g.pre) & 15u)))
    return LMOE_ERR_INVALID_ARG;
  // From here on the kernel counts K in units of 2 bytes: an e4m3 row of Kd codes is
  // addressed as Kd / 2 bf16-sized pairs, so tiles, boxes, swizzle and the gather offsets
  // are the same bytes for both operand types.
  GroupedArgs ga = g;
  const int kd = g.fp8 ? g.Kd / 2 : g.Kd;
  const int ld = g.fp8 ? x_ld / 2 : x_ld;
  ga.Kd = kd;
  if (g.fp8) ga.ldx = g.ldx / 2;
  CUtensorMap tw, tx;
  const uint64_t w_rows = static_cast<uint64_t>(g.E) * ceil_div(g.M_w, BLOCK_M) *
                          (kd / BLOCK_K) * BLOCK_M;  // tiled: rows of 128 bytes
  if (!make_tmap_bf16(&tw, W, w_rows, BLOCK_K, BLOCK_K, BLOCK_M) ||
      !make_tmap_bf16(&tx, X, x_rows, static_cast<uint64_t>(kd), static_cast<uint64_t>(ld),
                      GROUPED_BOX_T))
    return LMOE_ERR_CUDA;
  const bool shallow = g.epi != EPI_SITU && g.mean_tokens >= GROUPED_SHALLOW_MIN_TOKENS;
  // Each weight byte is read exactly once: marking it evict-first keeps the token rows, which
  // every weight row tile of an expert re-reads, in L2 (gate/value 1.20 -> 1.11 ms at the K3
  // prefill shape).  The down GEMM at prefill measured no gain (its output write-back shares
  // L2), so it keeps the default policy there.
  ga.evict_first = (g.epi == EPI_SITU || !shallow) ? 1 : 0;
  const bool wide = g.tokn > GROUPED_TOKN;
  // Weight-tile pairs when experts average many tokens (the token rows bound the shared-memory
  // fill), and at any load for a GEMM whose token rows come by TMA and whose outputs are bf16
  // (the down GEMM, the backward's dgrad GEMMs) and for the bf16 gate/value GEMM that keeps no
  // pre-activations: with about one token per expert (decode) a pair stage holds twice the
  // weight bytes of a single tile's, and its undivided accumulator drains in a few columns.
  // Decode (A/B, bit-identical outputs): down 0.354 -> 0.313 ms over SM pairs (e4m3 0.228 ->
  // 0.180 ms on one SM), gate/value 0.651 -> 0.630 ms.
  const bool pairs = g.mean_tokens >= GROUPED_PAIR_MIN_TOKENS ||
                     (!g.gather && g.epi == EPI_BF16) ||
                     (g.gather && g.epi == EPI_SITU && !g.pre && !g.fp8);
  if (g.fp8) {
    // e4m3 operands: pairs for the down GEMM only.  The gate/value GEMM's mainloop is half as
    // long as the bf16 one while its SiTU epilogue (the accurate tanh) is heavier, so the pair's
    // undivided accumulator, drained while no MMA runs, cost more than the token bytes saved
    // (prefill 0.634 -> 0.681 ms, skew 2.09 -> 2.74 ms; down 0.586 -> 0.564, 2.34 -> 1.91).
    if (pairs && g.epi != EPI_SITU && g.tokn <= GROUPED_TOKN_NARROW)
      // 128-token chunks (decode-like loads): two accumulator sets, so the drain, which bounds
      // this GEMM (its K is 512 codes: four K-blocks), runs under the next tile's MMAs
      return launch_grouped_stages<GROUPED_STAGES_PAIR + 1, true, 2, GROUPED_TOKN_NARROW>(
          tw, tx, ga, stream);
    if (pairs && g.epi != EPI_SITU) {
      if (wide) return launch_grouped_stages<GROUPED_STAGES_PAIR, true, 2, GROUPED_TOKN_WIDE>(
                    tw, tx, ga, stream);
      return launch_grouped_stages<GROUPED_STAGES_PAIR, true, 2, GROUPED_TOKN>(tw, tx, ga,
                                                                               stream);
    }
    if (wide) return launch_grouped_stages<GROUPED_STAGES_SHALLOW, true, 1, GROUPED_TOKN_WIDE>(
                  tw, tx, ga, stream);
    return shallow ? launch_grouped_stages<GROUPED_STAGES_SHALLOW, true, 1, GROUPED_TOKN>(
                         tw, tx, ga, stream)
                   : launch_grouped_stages<GROUPED_STAGES_DEEP, true, 1, GROUPED_TOKN>(
                         tw, tx, ga, stream);
  }
  // bf16 pairs (see above)
  if (pairs && !g.gather && g.epi == EPI_BF16 && GROUPED_SM_PAIR && g.M_w % (4 * BLOCK_M) == 0) {
    // ... over SM pairs, two weight tiles per SM, when the token rows come by TMA
    CUtensorMap tx16;
    if (!make_tmap_bf16(&tx16, X, x_rows, static_cast<uint64_t>(kd), static_cast<uint64_t>(ld),
                        GroupedPairCfg<4, GROUPED_TOKN_WIDE>::BOX_T))
      return LMOE_ERR_CUDA;
    if (wide) return launch_grouped_pair<4, GROUPED_TOKN_WIDE>(tw, tx16, x_rows, ga, stream);
    return launch_grouped_pair<4, GROUPED_TOKN>(tw, tx16, x_rows, ga, stream);
  }
  if (pairs) {
    if (wide) return launch_grouped_stages<GROUPED_STAGES_PAIR, false, 2, GROUPED_TOKN_WIDE>(
                  tw, tx, ga, stream);
    if (g.epi == EPI_SITU && !g.pre)  // no output staging: four stages
      return launch_grouped_stages<GROUPED_STAGES_PAIR + 1, false, 2, GROUPED_TOKN, false>(
          tw, tx, ga, stream);
    return launch_grouped_stages<GROUPED_STAGES_PAIR, false, 2, GROUPED_TOKN>(tw, tx, ga,
                                                                              stream);
  }
  if (wide) return launch_grouped_stages<GROUPED_STAGES_SHALLOW, false, 1, GROUPED_TOKN_WIDE>(
                tw, tx, ga, stream);
  return shallow ? launch_grouped_stages<GROUPED_STAGES_SHALLOW, false, 1, GROUPED_TOKN>(
                       tw, tx, ga, stream)
                 : launch_grouped_stages<GROUPED_STAGES_DEEP, false, 1, GROUPED_TOKN>(
                       tw, tx, ga, stream);
}

}  // namespace lmoe
