// kernels.cuh -- internal launchers and buffer layouts of the lmoe library.
#pragma once

#include <cuda.h>
#include <stddef.h>

#include "common.cuh"

namespace lmoe {

// Offsets (bytes) of the pieces of the packed weight buffer; every piece 1024-aligned.
struct PackedLayout {
  size_t w1, wr, wgu, wed, w2, gamma, total;
  size_t sgu, sed;  // e4m3 experts: per-row scales of wgu / wed
};

// Offsets (bytes) of the forward workspace; every buffer 256-aligned.
struct WorkspaceLayout {
  size_t err, lat, logits, logits_t, scores, tau, idx, gate, masks, base, offsets, ct_off, inv,
      src_tok, h, o, zh, ys;
  size_t ct_off2;             // a routed GEMM's own chunk prefix sum (gate/value or down)
  size_t lat8, slat, h8, sh;  // e4m3 experts: quantised latent and SiTU output, row scales
  size_t splitk;              // small batches: split-K partial sums of the dense GEMMs
  size_t total_base;          // bytes without the split-K region (which is optional)
  size_t total;               // bytes with it
};

PackedLayout packed_layout(const lmoe_dims& D);
WorkspaceLayout workspace_layout(const lmoe_dims& D);
// lmoe_forward's argument checks for T > 0 (LMOE_OK, or the status it would return).
int forward_args_check(const lmoe_dims* dims, const void* packed, const void* x,
                       const void* residual, const void* y, const void* workspace,
                       size_t ws_bytes, const lmoe_io* io);

// Epilogues of the tcgen05 GEMM.
enum EpiMode : int {
  EPI_BF16 = 0,   // out0[r, c] = bf16(acc)
  EPI_F32 = 1,    // outf[r, c] = acc
  EPI_SITU = 2,   // out1[r, c/2 + i] = bf16(SiTU(gate_i, value_i)) over 16+16 interleave
  EPI_SPLIT = 3,  // columns < split: EPI_BF16 to out0; others: EPI_SITU to out1 (c - split)
  EPI_RESID = 4   // out0[r, c] = bf16(acc + resid[r, c]) (resid may be null); with outf,
                  // also outf[r, c] = acc + resid[r, c] in fp32 (the value before rounding)
};

struct GemmArgs {
  int M;                  // rows of A and of the output
  int N;                  // output columns
  int Kd;                 // reduction length, multiple of 64
  int epi;
  int split;
  __nv_bfloat16* out0;
  int ld0;
  __nv_bfloat16* out1;
  int ld1;
  float* outf;
  int ldf;
  float* outf_t;          // EPI_F32: optional transposed copy, outf_t[c * ldt + r]
  int ldt;
  const float* col_bias;  // EPI_F32: optional per-column addend, outf[r, c] = acc + col_bias[c]
  const __nv_bfloat16* resid;
  int ldr;
  const float* addf;      // EPI_RESID: optional fp32 addend addf[r * lda + c]
  int lda;
  __nv_bfloat16* pre;     // EPI_SITU / EPI_SPLIT: optional bf16 copy of the gate/value
  int ldp;                // pre-activations, pre[r * ldp + c] (EPI_SPLIT: c - split)
  int max_ctas;           // persistent grid limit (0: one CTA per SM)
  float c;                // SiTU cap
  uint32_t* err;          // device error flag (never null)
  unsigned long long timeout_ns;
  int out_tma;            // set by launch_gemm: grouped-K output through tensor stores
  int inject_stall;       // test hook: the MMA role first waits on a barrier nobody arrives
                          // on, so every role runs into its bounded wait and aborts
  // Grouped-K mode (groups > 0): `groups` independent products C_q = A_q^T B_q with A and B
  // MN-major (token-major): A [rows, M] and B [rows, N] row-major, group q reducing over the
  // rows [kseg[q], kseg[q + 1]) (any boundaries; an empty range gives zeros; the rows of
  // the next group that a last K-block reaches are zeroed in A's tile, so B's must be
  // finite).  EPI_F32 only; group q's output at outf + q * group_stride, output row
  // row_map[r] (or r).
  int groups;
  const int32_t* kseg;
  long long group_stride;
  const int32_t* row_map;
  // groups == 1 whose range is every row [0, kfull) of A and B (kfull > 0; the caller knows
  // it on the host): such a product may run over SM pairs, reading no kseg
  int kfull;
  // Split-K (dense mode, set by the launcher when one M-tile leaves most SMs idle): slice s of
  // ksplit reduces its share of the K-blocks into partial[s, M, N] (fp32), and a second kernel
  // sums the slices in order and applies the epilogue.  partial: caller's scratch of
  // partial_bytes, or null (no split).
  int ksplit;
  float* partial;
  size_t partial_bytes;
  int* extra_launches;    // optional: incremented by the kernels launch_gemm enqueues beyond
                          // the GEMM itself (the split-K sum)
};
constexpr size_t SPLITK_BYTES = size_t{12} << 20;  // workspace for split-K partials (T <= 128)

// Routed-expert GEMMs (gemm_grouped.cu): out[tok, r] = act[tok, :] . W[e][r, :] for the
// token rows of each expert segment, weight rows on the MMA's M side.
struct GroupedArgs {
  int E;                  // experts
  int M_w;                // weight rows per expert (2I for gate/value, L for down)
  int Kd;                 // reduction length (L for gate/value, I for down), multiple of 64
                          // (of 128 with fp8)
  const int32_t* seg_off; // [E+1] first token row of each expert's segment
  const int32_t* ct_off;  // [E+1] prefix sum of ceil(count / tokn)
  int tokn;               // chunk granularity ct_off was built with (grouped_tokn)
  const int32_t* gather;  // [rows] source row of each permuted row, or null: then the
                          // activation rows are the permuted rows themselves (TMA boxes)
  const __nv_bfloat16* x; // gathered activations [*, ldx] (with gather)
  int ldx;
  int epi;                // EPI_SITU (gate/value, M_w = 2I) or EPI_BF16
  __nv_bfloat16* out;     // [rows, ldo] token-major output
  int ldo;
  float c;
  uint32_t* err;
  unsigned long long timeout_ns;
  int max_ctas;           // persistent grid limit (0: one CTA per SM)
  int mean_tokens;        // average tokens per expert (T*K/E): picks the pipeline depth
  int evict_first;        // set by the launcher: weights loaded with an L2 evict-first policy
  int out_tma;            // set by the launcher: whole 32-token output chunks by tensor stores
  // e4m3 operands: W and x hold codes, Kd and ldx count codes, a K-block is 128 codes (the
  // same 128 bytes per row as 64 bf16); the accumulator is multiplied by the weight row's
  // and the activation row's scale in the epilogue
  int fp8;
  const float* w_scale;   // [E * ceil(M_w / 128) * 128] per weight row
  const float* x_scale;   // per activation row, indexed like the rows (through gather)
  // EPI_SITU: also store the bf16 pre-activations, pre[row, weight row] (row stride ldp)
  __nv_bfloat16* pre;
  int ldp;
};

// W: the experts' weights in tiles of 128 rows x 128 bytes (64 bf16 or 128 e4m3 codes),
// ordered (expert, row tile, column tile).
int launch_grouped_gemm(const void* W, const void* X, uint64_t x_rows, int x_ld,
                        const GroupedArgs& g, cudaStream_t stream);

// Encodes a 2-D bf16 row-major [rows, cols] (row stride ld elements) TMA map with a
// 64 x box_rows box and the 128-byte swizzle.  Returns false on failure.
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                    uint32_t box_rows);
bool make_tmap_bf16_out32(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                          uint64_t ld);

int launch_gemm(const void* A, uint64_t a_rows, int a_ld, const void* B, uint64_t b_rows,
                int b_ld, const GemmArgs& args, cudaStream_t stream);

// Top-K routing of [T, E] logits, or with scores of the router scores themselves.
int launch_route(const float* logits, const float* tau, int T, int E, int K, int32_t* idx,
                 float* gate, float* scores_out, bool scores, cudaStream_t stream);
// Thresholds from logits (or, with scores, router scores) stored with element (t, e) at
// z[t * stride_t + e * stride_e] (stride_t = 1, stride_e = T is the fast, expert-major
// layout).
int launch_thresholds(const float* z, int T, int E, int64_t stride_t, int64_t stride_e, int k,
                      float* tau, bool scores, cudaStream_t stream);
// Router scores of [T, E] logits z: s[T, E] and, if s_t is given, the expert-major s_t[E, T].
int launch_scores(const float* z, int T, int E, float* s, float* s_t, cudaStream_t stream);
// Per expert, the logits of the min(k, T) largest scores (rows of cand, stride ldc), then
// -FLT_MAX up to row k.
int launch_candidates(const float* z, int T, int E, int64_t stride_t, int64_t stride_e, int k,
                      float* cand, int64_t ldc, cudaStream_t stream);
// out[E, T] = in[T, E]^T (fp32).
int launch_transpose_f32(const float* in, int T, int E, float* out, cudaStream_t stream);
// Checked mode: sets DEVERR_NONFINITE in *err if any of p[0, n) is NaN or infinite.
int launch_finite_check(const float* p, int64_t n, uint32_t* err, cudaStream_t stream);
// ct_off: prefix sums of ceil(count / tokn) (tokn = grouped_tokn of the batch); ct_off2, if
// not null: the same for tokn2.
int launch_dispatch(const int32_t* idx, int T, int E, int K, uint32_t* masks, uint32_t* base,
                    int32_t* offsets, int32_t* ct_off, int tokn, int32_t* ct_off2, int tokn2,
                    int32_t* inv, int32_t* src_tok, int32_t* counts_out, uint32_t* err,
                    cudaStream_t stream);
int launch_combine(const __nv_bfloat16* o, const float* gate, const int32_t* inv,
                   const float* gamma, int T, int K, int L, float eps, __nv_bfloat16* z,
                   int ldz, uint32_t* err, unsigned long long timeout_ns, cudaStream_t stream);
// Streaming thresholds: tau_ema = first ? tau_step : fma(beta, tau_ema - tau_step, tau_step).
int launch_tau_ema(const float* tau_step, float* tau_ema, int E, float beta, int first,
                   cudaStream_t stream);
// Load counters (layout at lmoe_load_stats_update) from counts, or from segment offsets.
int launch_load_stats(const int32_t* counts, const int32_t* offsets, int E,
                      unsigned long long* acc, cudaStream_t stream);
// Expert-parallel dispatch / combine over R ranks (see ep.cu); ws: ep_workspace_bytes.
size_t ep_workspace_bytes(int T, int R);
int launch_ep_dispatch(const int32_t* idx, int T, int K, int E, int R, const void* rows, int W,
                       void* send_rows, int32_t* send_off, int32_t* send_tok,
                       uint32_t* send_slots, void* ws, cudaStream_t stream);
int launch_ep_combine(const int32_t* idx, int T, int K, int E, int R, const int32_t* send_off,
                      const int32_t* send_tok, const uint32_t* send_slots, const int32_t* inv,
                      const float* gate, const void* o, int W, void* part, float* u,
                      const void* ws, cudaStream_t stream);
// Transposed tiled expert weights for the backward pass (pack.cu).
int launch_pack_backward(const lmoe_dims& D, const lmoe_weights& w, __nv_bfloat16* wgu_t,
                         __nv_bfloat16* wed_t, cudaStream_t stream);
// Backward of the routed branch (bwd.cu).
int launch_combine_bwd(const __nv_bfloat16* o, const float* gate, const int32_t* inv,
                       const float* gamma, const float* dz, int T, int K, int L, float eps,
                       __nv_bfloat16* dout, float* dgate, float* u, float* r, uint32_t* err,
                       unsigned long long timeout_ns, cudaStream_t stream);
int launch_dgamma(const float* dz, const float* u, const float* r, int T, int L, float* part,
                  float* dgamma, cudaStream_t stream);
int launch_situ_bwd(const __nv_bfloat16* pre, const __nv_bfloat16* dh, int64_t rows, int I,
                    float c, __nv_bfloat16* dgv, int64_t ldo, cudaStream_t stream);
int launch_slot_sum(const __nv_bfloat16* x, const int32_t* inv, int T, int K, int L,
                    const float* add, float* out, __nv_bfloat16* outb, int64_t ldb,
                    cudaStream_t stream);
int launch_gather_rows(const __nv_bfloat16* x, int64_t ldx, const int32_t* idx, int64_t n, int W,
                       __nv_bfloat16* out, int64_t ldo, cudaStream_t stream);
int launch_rowmap(int I, int base, int32_t* map, int32_t* seg, int seg_len, cudaStream_t stream);
// Router backward: dz [T, ldo] bf16 from the logits z [T, ldz], routing and dgate.
int launch_router_bwd(const float* z, int64_t ldz, const int32_t* idx, const float* gate,
                      const float* dgate, int T, int K, __nv_bfloat16* dz, int ldo,
                      cudaStream_t stream);
// xt[w, q] = x[q, w] for q < n, zero up to qmax (a multiple of 64).
int launch_transpose_rows(const __nv_bfloat16* x, int64_t ldx, int W, int64_t n, int64_t qmax,
                          int64_t ldt, __nv_bfloat16* xt, cudaStream_t stream);
// Per-row e4m3 quantisation of bf16 rows (cols % 16 == 0): codes [rows, ldq], scales [rows].
int launch_quantize_rows(const __nv_bfloat16* x, int64_t rows, int cols, int64_t ldx,
                         uint8_t* q, int64_t ldq, float* scales, cudaStream_t stream);
// Expert weights -> e4m3 tiles of 128 rows x 128 codes + per-row scales (see quant.cu).
int launch_pack_tiled_e4m3(uint8_t* dst, float* scales, const __nv_bfloat16* w,
                           const __nv_bfloat16* w_g, const __nv_bfloat16* w_v, int glu, int E,
                           int M_w, int Kd, cudaStream_t stream);
int launch_pack(const lmoe_dims& D, const lmoe_weights& w, const PackedLayout& P, uint8_t* base,
                cudaStream_t stream);

}  // namespace lmoe
