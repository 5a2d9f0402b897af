// api.cu -- the extern "C" entry points declared in include/lmoe.h: argument checks,
// buffer layouts, and the sequence of kernel launches of one forward pass.
#include <stdlib.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

// Per-stage NVTX ranges ("lmoe" domain, one range per stage of lmoe_forward around the
// launches of that stage), so that a profiler can attribute and filter kernels by stage
// (ncu --nvtx --nvtx-include "lmoe@expert_gate_up/").  Without an attached tool the NVTX
// calls return at once.
static const char* const STAGE_NAMES[LMOE_NUM_STAGES] = {
    "latent_shared", "router", "thresholds", "route", "dispatch",
    "expert_gate_up", "expert_down", "combine", "output"};

static nvtxDomainHandle_t nvtx_domain() {
  static nvtxDomainHandle_t d = nvtxDomainCreateA("lmoe");
  return d;
}

class StageRanges {
 public:
  ~StageRanges() { close(); }
  // ends the open stage's range and opens `stage`'s (none for LMOE_NUM_STAGES)
  void enter(int stage) {
    close();
    if (stage < 0 || stage >= LMOE_NUM_STAGES) return;
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = STAGE_NAMES[stage];
    nvtxDomainRangePushEx(nvtx_domain(), &a);
    open_ = true;
  }

 private:
  void close() {
    if (open_) nvtxDomainRangePop(nvtx_domain());
    open_ = false;
  }
  bool open_ = false;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static bool dims_ok(const lmoe_dims* D) {
  if (!D) return false;
  if (D->T < 0 || D->d <= 0 || D->L <= 0 || D->E <= 0 || D->K <= 0 || D->I <= 0 || D->S < 0 ||
      D->Is < 0)
    return false;
  if (!(D->c > 0.0f) || !(D->eps >= 0.0f)) return false;
  if (D->expert_fp8 != 0 && D->expert_fp8 != 1) return false;
  return true;
}

static int dims_supported(const lmoe_dims* D) {
  if (!dims_ok(D)) return LMOE_ERR_INVALID_ARG;
  if (D->d % 64 || D->L % 64 || D->I % 64) return LMOE_ERR_UNSUPPORTED;
  if (D->S > 0 && (D->Is <= 0 || D->Is % 64)) return LMOE_ERR_UNSUPPORTED;
  if (D->K > D->E || D->K > 32 || D->E > 4096 || D->E % 16) return LMOE_ERR_UNSUPPORTED;
  if (D->L > 16384) return LMOE_ERR_UNSUPPORTED;
  if (D->expert_fp8 && (D->L % 128 || D->I % 128)) return LMOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(D->T) * D->K >= (int64_t{1} << 31)) return LMOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(D->E) * 2 * D->I >= (int64_t{1} << 31) ||
      static_cast<int64_t>(D->E) * D->L >= (int64_t{1} << 31))
    return LMOE_ERR_UNSUPPORTED;
  return LMOE_OK;
}

static int shared_width(const lmoe_dims& D) { return D.S > 0 ? D.S * D.Is : 0; }

PackedLayout packed_layout(const lmoe_dims& D) {
  PackedLayout P{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes, 1024);
    return o;
  };
  const size_t sw = static_cast<size_t>(shared_width(D));
  P.w1 = take((static_cast<size_t>(D.L) + 2 * sw) * D.d * 2);
  P.wr = take(static_cast<size_t>(D.E) * D.L * 2);
  // expert weights in 128-row tiles (the last row tile of an expert zero-padded): bf16, or
  // e4m3 codes (one byte each) with one fp32 scale per row
  const size_t eb = D.expert_fp8 ? 1 : 2;
  const size_t rows_gu = static_cast<size_t>(D.E) * ceil_div(2 * D.I, BLOCK_M) * BLOCK_M;
  const size_t rows_ed = static_cast<size_t>(D.E) * ceil_div(D.L, BLOCK_M) * BLOCK_M;
  P.wgu = take(rows_gu * D.L * eb);
  P.wed = take(rows_ed * D.I * eb);
  P.w2 = take(static_cast<size_t>(D.d) * (D.L + sw) * 2);
  P.gamma = take(static_cast<size_t>(D.L) * 4);
  P.sgu = P.sed = 0;
  if (D.expert_fp8) {
    P.sgu = take(rows_gu * 4);
    P.sed = take(rows_ed * 4);
  }
  P.total = off;
  return P;
}

WorkspaceLayout workspace_layout(const lmoe_dims& D) {
  WorkspaceLayout W{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return o;
  };
  const size_t T = static_cast<size_t>(D.T), TK = T * D.K;
  const size_t nb = static_cast<size_t>(ceil_div(D.T, DISPATCH_TOKENS));
  W.err = take(256);  // word 0: device error flag; word 1: dispatch scan completion counter
  W.lat = take(T * D.L * 2);
  W.logits = take(T * D.E * 4);
  W.logits_t = take(T * D.E * 4);
  W.scores = take(T * D.E * 4);
  W.tau = take(static_cast<size_t>(D.E) * 4);
  W.idx = take(TK * 4);
  W.gate = take(TK * 4);
  W.masks = take(nb * D.E * 4);
  W.base = take(nb * D.E * 4);
  W.offsets = take((static_cast<size_t>(D.E) + 1) * 4);
  W.ct_off = take((static_cast<size_t>(D.E) + 1) * 4);
  W.ct_off2 = take((static_cast<size_t>(D.E) + 1) * 4);
  W.inv = take(TK * 4);
  W.src_tok = take(TK * 4);
  W.h = take(TK * D.I * 2);
  W.o = take(TK * D.L * 2);
  W.zh = take(T * (D.L + shared_width(D)) * 2);
  // fp32 shared-expert output, used when the shared experts run beside the routed path
  W.ys = take(D.T >= LMOE_OVERLAP_MIN_T && shared_width(D) > 0 ? T * D.d * 4 : 0);
  W.lat8 = W.slat = W.h8 = W.sh = 0;
  if (D.expert_fp8) {
    W.lat8 = take(T * D.L);
    W.slat = take(T * 4);
    W.h8 = take(TK * D.I);
    W.sh = take(TK * 4);
  }
  W.total_base = off;
  // small batches: room for split-K partial sums of the dense GEMMs (optional; lmoe_forward
  // splits only when the caller's workspace includes it)
  W.splitk = off;
  if (D.T > 0 && D.T <= BLOCK_M) take(SPLITK_BYTES);
  W.total = off;
  return W;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static uint64_t wait_limit_ns() {
  // Upper bound of any single device-side wait.  Legitimate waits last microseconds.
  const char* s = getenv("LMOE_WAIT_LIMIT_MS");
  if (s && *s) {
    const long v = strtol(s, nullptr, 10);
    if (v > 0 && v < 60000) return static_cast<uint64_t>(v) * 1000000ull;
  }
  return 2000ull * 1000000ull;
}

// Test hook: LMOE_FAULT_INJECT=stall makes the first GEMM of each call wait on a barrier
// that nothing arrives on, so the bounded-wait error path can be exercised without any
// fault.  Read at every call.
static bool inject_stall() {
  const char* s = getenv("LMOE_FAULT_INJECT");
  return s && strcmp(s, "stall") == 0;
}

// Checked mode: LMOE_CHECK_FINITE=1 makes lmoe_forward scan the router logits; a
// non-finite one is reported as an invalid argument by lmoe_last_device_error.  Read at
// every call.
static bool check_finite() {
  const char* s = getenv("LMOE_CHECK_FINITE");
  return s && strcmp(s, "1") == 0;
}

static GemmArgs gemm_defaults(uint32_t* err, float c) {
  GemmArgs g{};
  g.err = err;
  g.c = c;
  g.timeout_ns = wait_limit_ns();
  return g;
}

// Backward of the routed branch: transposed expert weights and scratch.
struct BwdPacked {
  size_t wgu_t, wed_t;       // expert weights transposed, in 128-row tiles
  size_t wout_t, wr_t, wls_t;  // dense weights transposed (whole-layer backward)
  size_t total;
};
static int pad64(int n) { return (n + 63) / 64 * 64; }
static BwdPacked bwd_packed_layout(const lmoe_dims& D) {
  BwdPacked B{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes, 1024);
    return o;
  };
  B.wgu_t = take(static_cast<size_t>(D.E) * ceil_div(D.L, BLOCK_M) * BLOCK_M * 2 * D.I * 2);
  B.wed_t = take(static_cast<size_t>(D.E) * ceil_div(D.I, BLOCK_M) * BLOCK_M * D.L * 2);
  const size_t sw = static_cast<size_t>(D.S > 0 ? D.S * D.Is : 0);
  B.wout_t = take((D.L + sw) * D.d * 2);                       // [L + sw, d]
  B.wr_t = take(static_cast<size_t>(D.L) * pad64(D.E) * 2);      // [L, E padded to 64]
  B.wls_t = take(static_cast<size_t>(D.d) * (D.L + 2 * sw) * 2);  // [d, L + 2 sw]
  B.total = off;
  return B;
}

struct BwdLayout {
  size_t u, r, dout, dh, pre, dgv, dlatp, part, rowmap, latp, total;
};
static BwdLayout bwd_layout(const lmoe_dims& D) {
  BwdLayout B{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return o;
  };
  const size_t T = static_cast<size_t>(D.T), TK = T * D.K, L = D.L, I = D.I;
  B.u = take(T * L * 4);
  B.r = take(T * 4);
  B.dout = take(TK * L * 2);
  B.dh = take(TK * I * 2);
  B.pre = take(TK * 2 * I * 2);
  B.dgv = take(TK * 2 * I * 2);
  B.dlatp = take(TK * L * 2);
  B.part = take(64 * L * 4);
  B.rowmap = take(2 * I * 4);
  B.latp = take(TK * L * 2);
  B.total = off;
  return B;
}

// The whole layer's backward adds these buffers after the routed branch's.
struct LayerBwdLayout {
  size_t dz, dhs, dgate, dlogit, dlat_r, dlat, dcat, pre_s, seg1, rowmap_s, total;
  int Ep, sw, wc, wz;  // E padded to 64; shared width; widths of dcat and zh
};
static LayerBwdLayout layer_bwd_layout(const lmoe_dims& D) {
  LayerBwdLayout B{};
  size_t off = bwd_layout(D).total;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return o;
  };
  B.Ep = pad64(D.E);
  B.sw = D.S > 0 ? D.S * D.Is : 0;
  B.wc = D.L + 2 * B.sw;
  B.wz = D.L + B.sw;
  const size_t T = static_cast<size_t>(D.T), L = D.L;
  B.dz = take(T * L * 4);
  B.dhs = take(T * B.sw * 2);
  B.dgate = take(T * D.K * 4);
  B.dlogit = take(T * B.Ep * 2);
  B.dlat_r = take(T * L * 4);
  B.dlat = take(T * L * 4);
  B.dcat = take(T * B.wc * 2);
  B.pre_s = take(T * 2 * B.sw * 2);
  B.seg1 = take(2 * 4);
  B.rowmap_s = take(static_cast<size_t>(B.wc) * 4);
  B.total = off;
  return B;
}

// The routed branch's backward in two halves, shared by lmoe_routed_backward and
// lmoe_backward (which runs the router's backward between them).
struct RoutedBwd {
  lmoe_dims D;
  const uint8_t* pk;  // packed forward weights
  const uint8_t* pb;  // packed transposed weights
  uint8_t* ws;        // forward workspace (the batch's routing and activations)
  uint8_t* bw;        // backward workspace
  PackedLayout P;
  BwdPacked PB;
  WorkspaceLayout W;
  BwdLayout B;
  cudaStream_t stream;
  const __nv_bfloat16* pre;  // the forward's saved pre-activations, or null: recompute
};

// 1-2. RMSNorm and combine backward (du, do_j, dgate_j), then dgamma.
static int routed_bwd_front(const RoutedBwd& R, const float* dz, float* dgate, float* dgamma) {
  using bf = __nv_bfloat16;
  const lmoe_dims& D = R.D;
  int rc = launch_combine_bwd(reinterpret_cast<const bf*>(R.ws + R.W.o),
                              reinterpret_cast<const float*>(R.ws + R.W.gate),
                              reinterpret_cast<const int32_t*>(R.ws + R.W.inv),
                              reinterpret_cast<const float*>(R.pk + R.P.gamma), dz, D.T, D.K, D.L,
                              D.eps, reinterpret_cast<bf*>(R.bw + R.B.dout), dgate,
                              reinterpret_cast<float*>(R.bw + R.B.u),
                              reinterpret_cast<float*>(R.bw + R.B.r),
                              reinterpret_cast<uint32_t*>(R.ws + R.W.err), wait_limit_ns(),
                              R.stream);
  if (rc != LMOE_OK) return rc;
  return launch_dgamma(dz, reinterpret_cast<const float*>(R.bw + R.B.u),
                       reinterpret_cast<const float*>(R.bw + R.B.r), D.T, D.L,
                       reinterpret_cast<float*>(R.bw + R.B.part), dgamma, R.stream);
}


}  // namespace lmoe

using namespace lmoe;

// 3-11. dgrad through the experts (dlat, plus `dlat_add` when given, also copied to bf16
// into dlat_b with row stride ldb when given), then the expert weight gradients.
static int routed_bwd_back(const RoutedBwd& R, const float* dlat_add, float* dlat,
                           __nv_bfloat16* dlat_b, int64_t ldb, float* dw_gu, float* dw_ed) {
  using bf = __nv_bfloat16;
  const lmoe_dims& D = R.D;
  const int T = D.T, K = D.K, L = D.L, I = D.I, E = D.E, TK = T * K;
  const WorkspaceLayout& W = R.W;
  const BwdLayout& B = R.B;
  const PackedLayout& P = R.P;
  const BwdPacked& PB = R.PB;
  const uint8_t* pk = R.pk;
  const uint8_t* pb = R.pb;
  uint8_t* ws = R.ws;
  uint8_t* bw = R.bw;
  cudaStream_t stream = R.stream;
  uint32_t* err = reinterpret_cast<uint32_t*>(ws + W.err);
  const int32_t* offsets = reinterpret_cast<const int32_t*>(ws + W.offsets);
  const int32_t* ct_off = reinterpret_cast<const int32_t*>(ws + W.ct_off);
  const int32_t* inv = reinterpret_cast<const int32_t*>(ws + W.inv);
  const int32_t* src_tok = reinterpret_cast<const int32_t*>(ws + W.src_tok);
  const bf* lat = reinterpret_cast<const bf*>(ws + W.lat);
  const bf* h = reinterpret_cast<const bf*>(ws + W.h);
  bf* dout = reinterpret_cast<bf*>(bw + B.dout);
  bf* dh = reinterpret_cast<bf*>(bw + B.dh);
  bf* pre = reinterpret_cast<bf*>(bw + B.pre);
  bf* dgv = reinterpret_cast<bf*>(bw + B.dgv);
  bf* dlatp = reinterpret_cast<bf*>(bw + B.dlatp);
  int32_t* rowmap = reinterpret_cast<int32_t*>(bw + B.rowmap);
  int rc;
  auto grouped = [&](int M_w, int Kd, const int32_t* gather, const bf* x, int ldx, int epi,
                     bf* out, int ldo) {
    GroupedArgs g{};
    g.E = E;
    g.M_w = M_w;
    g.Kd = Kd;
    g.seg_off = offsets;
    g.ct_off = ct_off;
    g.gather = gather;
    g.x = x;
    g.ldx = ldx;
    g.epi = epi;
    g.out = out;
    g.ldo = ldo;
    g.c = D.c;
    g.err = err;
    g.timeout_ns = wait_limit_ns();
    g.mean_tokens = static_cast<int>(static_cast<int64_t>(TK) / E);
    g.tokn = grouped_tokn(T, D.K, E);  // as the forward's dispatch built ct_off
    return g;
  };
  // 3. dh = do . W_ed (per expert, weights transposed)
  {
    GroupedArgs g = grouped(I, L, nullptr, nullptr, 0, EPI_BF16, dh, I);
    if ((rc = launch_grouped_gemm(pb + PB.wed_t, dout, static_cast<uint64_t>(TK), L, g, stream)) !=
        LMOE_OK)
      return rc;
  }
  // 4. gate/value pre-activations (interleaved rows): the forward's, or computed again;
  // 5. through SiTU
  const bf* pre_in = R.pre;
  if (!pre_in) {
    GroupedArgs g = grouped(2 * I, L, src_tok, lat, L, EPI_BF16, pre, 2 * I);
    if ((rc = launch_grouped_gemm(pk + P.wgu, lat, static_cast<uint64_t>(T), L, g, stream)) !=
        LMOE_OK)
      return rc;
    pre_in = pre;
  }
  if ((rc = launch_situ_bwd(pre_in, dh, TK, I, D.c, dgv, 2 * I, stream)) != LMOE_OK) return rc;
  // 6. dlat_p = dgv . W_gu (per expert, weights transposed), 7. summed over the slots
  {
    GroupedArgs g = grouped(L, 2 * I, nullptr, nullptr, 0, EPI_BF16, dlatp, L);
    if ((rc = launch_grouped_gemm(pb + PB.wgu_t, dgv, static_cast<uint64_t>(TK), 2 * I, g,
                                  stream)) != LMOE_OK)
      return rc;
  }
  if ((rc = launch_slot_sum(dlatp, inv, T, K, L, dlat_add, dlat, dlat_b, ldb, stream)) != LMOE_OK) return rc;
  // 8. the latent rows in slot order (the weight gradient's B operand); output rows of the
  // packed gate/value rows
  bf* latp = reinterpret_cast<bf*>(bw + B.latp);
  if ((rc = launch_gather_rows(lat, L, src_tok, TK, L, latp, L, stream)) != LMOE_OK ||
      (rc = launch_rowmap(I, 0, rowmap, nullptr, 0, stream)) != LMOE_OK)
    return rc;
  // 9. dW_ed[e] = do_e^T h_e   [L, I];  10. dW_gu[e] = dgv_e^T lat_e   [2I, L] (gate rows,
  // then value rows): each over its expert's slot rows, operands read token-major
  {
    GemmArgs g = gemm_defaults(err, D.c);
    g.M = L;
    g.N = I;
    g.epi = EPI_F32;
    g.outf = dw_ed;
    g.ldf = I;
    g.groups = E;
    g.kseg = offsets;
    g.group_stride = static_cast<long long>(L) * I;
    if ((rc = launch_gemm(dout, static_cast<uint64_t>(TK), L, h, static_cast<uint64_t>(TK), I, g,
                          stream)) != LMOE_OK)
      return rc;
  }
  {
    GemmArgs g = gemm_defaults(err, D.c);
    g.M = 2 * I;
    g.N = L;
    g.epi = EPI_F32;
    g.outf = dw_gu;
    g.ldf = L;
    g.groups = E;
    g.kseg = offsets;
    g.group_stride = static_cast<long long>(2 * I) * L;
    g.row_map = rowmap;
    if ((rc = launch_gemm(dgv, static_cast<uint64_t>(TK), 2 * I, latp, static_cast<uint64_t>(TK),
                          L, g, stream)) != LMOE_OK)
      return rc;
  }
  return LMOE_OK;
}


extern "C" {

const char* lmoe_error_string(int status) {
  switch (status) {
    case LMOE_OK: return "ok";
    case LMOE_ERR_INVALID_ARG: return "invalid argument";
    case LMOE_ERR_UNSUPPORTED: return "unsupported shape";
    case LMOE_ERR_CUDA: return "CUDA call or kernel launch failed";
    case LMOE_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out of time";
    case LMOE_ERR_WORKSPACE_TOO_SMALL: return "workspace or packed buffer too small";
    default: return "unknown status";
  }
}

const char* lmoe_version(void) { return "lmoe 0.1 sm_103a"; }

size_t lmoe_packed_bytes(const lmoe_dims* dims) {
  if (dims_supported(dims) != LMOE_OK) return 0;
  return packed_layout(*dims).total;
}

size_t lmoe_workspace_bytes(const lmoe_dims* dims) {
  if (dims_supported(dims) != LMOE_OK) return 0;
  return workspace_layout(*dims).total;
}

int lmoe_pack_weights(const lmoe_dims* dims, const lmoe_weights* w, void* packed,
                      size_t packed_bytes, void* stream) {
  const int rc = dims_supported(dims);
  if (rc != LMOE_OK) return rc;
  if (!w || !packed || !w->w_down || !w->w_router || !w->w_gate || !w->w_value || !w->w_edown ||
      !w->gamma || !w->w_up)
    return LMOE_ERR_INVALID_ARG;
  if (dims->S > 0 && (!w->w_sgate || !w->w_svalue || !w->w_sdown)) return LMOE_ERR_INVALID_ARG;
  const void* ptrs[] = {packed,  w->w_down,  w->w_router, w->w_gate,   w->w_value,
                        w->w_edown, w->gamma, w->w_up};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LMOE_ERR_INVALID_ARG;
  if (dims->S > 0 && (!aligned16(w->w_sgate) || !aligned16(w->w_svalue) || !aligned16(w->w_sdown)))
    return LMOE_ERR_INVALID_ARG;
  const PackedLayout P = packed_layout(*dims);
  if (packed_bytes < P.total) return LMOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_pack(*dims, *w, P, static_cast<uint8_t*>(packed),
                     static_cast<cudaStream_t>(stream));
}

int lmoe_fair_share_rank(long long T, int K, int E) {
  if (K < 1 || E < 1 || T < 0 || T > (static_cast<long long>(1) << 40)) return -1;
  if (T == 0) return 0;
  const long long f = T * K / E;
  return static_cast<int>(f < 1 ? 1 : (f > T ? T : f));
}

int lmoe_thresholds(const float* logits, int T, int E, int K, int k_rank, float* tau,
                    void* stream) {
  if (T < 0 || E < 1 || K < 1 || k_rank > T) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!logits || !tau) return LMOE_ERR_INVALID_ARG;
  const int k = k_rank > 0 ? k_rank : lmoe_fair_share_rank(T, K, E);
  // token-major input: each expert's column is read with stride E
  return launch_thresholds(logits, T, E, E, 1, k, tau, false, static_cast<cudaStream_t>(stream));
}

int lmoe_quantize_e4m3(const void* x, long long rows, int cols, uint8_t* codes, float* scales,
                       void* stream) {
  if (rows < 0 || cols <= 0) return LMOE_ERR_INVALID_ARG;
  if (rows == 0) return LMOE_OK;
  if (!x || !codes || !scales) return LMOE_ERR_INVALID_ARG;
  if (cols % 16 || !aligned16(x) || !aligned16(codes)) return LMOE_ERR_UNSUPPORTED;
  return launch_quantize_rows(static_cast<const __nv_bfloat16*>(x), rows, cols, cols, codes,
                              cols, scales, static_cast<cudaStream_t>(stream));
}

int lmoe_tau_ema(const float* tau_step, float* tau_ema, int E, float beta, int first,
                 void* stream) {
  if (E < 0 || !(beta >= 0.0f && beta <= 1.0f)) return LMOE_ERR_INVALID_ARG;
  if (E == 0) return LMOE_OK;
  if (!tau_step || !tau_ema) return LMOE_ERR_INVALID_ARG;
  return launch_tau_ema(tau_step, tau_ema, E, beta, first ? 1 : 0,
                        static_cast<cudaStream_t>(stream));
}

int lmoe_load_stats_update(const int32_t* counts, int E, unsigned long long* acc, void* stream) {
  if (E < 1 || !counts || !acc) return LMOE_ERR_INVALID_ARG;
  return launch_load_stats(counts, nullptr, E, acc, static_cast<cudaStream_t>(stream));
}

static int ep_args_ok(int T, int K, int E, int R) {
  if (T < 0 || K < 1 || E < 1 || R < 1) return LMOE_ERR_INVALID_ARG;
  if (K > 32 || R > 64 || E % R) return LMOE_ERR_UNSUPPORTED;
  return LMOE_OK;
}

size_t lmoe_ep_workspace_bytes(int T, int K, int E, int R) {
  if (ep_args_ok(T, K, E, R) != LMOE_OK) return 0;
  return ep_workspace_bytes(T, R) + 256;
}

int lmoe_ep_dispatch(const int32_t* idx, int T, int K, int E, int R, const void* rows, int W,
                     void* send_rows, int32_t* send_off, int32_t* send_tok, uint32_t* send_slots,
                     void* ws, size_t ws_bytes, void* stream) {
  int rc = ep_args_ok(T, K, E, R);
  if (rc != LMOE_OK) return rc;
  if (!send_off || (T > 0 && (!idx || !send_tok || !send_slots || !ws))) return LMOE_ERR_INVALID_ARG;
  if (rows && (!send_rows || W <= 0 || W % 8 || !aligned16(rows) || !aligned16(send_rows)))
    return LMOE_ERR_INVALID_ARG;
  if (ws_bytes < ep_workspace_bytes(T, R)) return LMOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0)
    return cudaMemsetAsync(send_off, 0, sizeof(int32_t) * (R + 1), st) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  return launch_ep_dispatch(idx, T, K, E, R, rows, rows ? W : 0, send_rows, send_off, send_tok,
                            send_slots, ws, st);
}

int lmoe_ep_combine(const int32_t* idx, int T, int K, int E, int R, const int32_t* send_off,
                    const int32_t* send_tok, const uint32_t* send_slots, const int32_t* inv,
                    const float* gate, const void* o, int W, void* part, float* u,
                    const void* ws, void* stream) {
  int rc = ep_args_ok(T, K, E, R);
  if (rc != LMOE_OK) return rc;
  if (T == 0) return LMOE_OK;
  if (!idx || !send_off || !send_tok || !send_slots || !inv || !gate || !o || !part || !u || !ws)
    return LMOE_ERR_INVALID_ARG;
  if (W <= 0 || W % 8 || !aligned16(o) || !aligned16(part) || !aligned16(u))
    return LMOE_ERR_INVALID_ARG;
  return launch_ep_combine(idx, T, K, E, R, send_off, send_tok, send_slots, inv, gate, o, W, part,
                           u, ws, static_cast<cudaStream_t>(stream));
}

int lmoe_threshold_candidates(const float* logits, int T, int E, int k, float* cand,
                              void* stream) {
  if (T < 0 || E < 1 || k < 1 || !cand || (T > 0 && !logits)) return LMOE_ERR_INVALID_ARG;
  // token-major input: each expert's column is read with stride E
  return launch_candidates(logits, T, E, E, 1, k, cand, E, static_cast<cudaStream_t>(stream));
}

int lmoe_route(const float* logits, const float* tau, int T, int E, int K, int32_t* idx,
               float* gate, float* scores_out, void* stream) {
  if (T < 0 || E < 1 || K < 1) return LMOE_ERR_INVALID_ARG;
  if (K > E || K > 32 || E > 4096) return LMOE_ERR_UNSUPPORTED;
  if (T == 0) return LMOE_OK;
  if (!logits || !idx || !gate) return LMOE_ERR_INVALID_ARG;
  return launch_route(logits, tau, T, E, K, idx, gate, scores_out, false,
                      static_cast<cudaStream_t>(stream));
}

int lmoe_gemm_bf16(const void* A, const void* B, float* C, int M, int N, int Kd,
                   uint32_t* dev_flag, void* stream) {
  if (M < 0 || N <= 0 || Kd <= 0 || !C || !A || !B || !dev_flag) return LMOE_ERR_INVALID_ARG;
  if (N % 16 || Kd % 64) return LMOE_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return LMOE_ERR_INVALID_ARG;
  if (M == 0) return LMOE_OK;
  GemmArgs g = gemm_defaults(dev_flag, 1.0f);
  g.M = M;
  g.N = N;
  g.Kd = Kd;
  g.epi = EPI_F32;
  g.outf = C;
  g.ldf = N;
  return launch_gemm(A, static_cast<uint64_t>(M), Kd, B, static_cast<uint64_t>(N), Kd, g,
                     static_cast<cudaStream_t>(stream));
}

int lmoe_gemm_wgrad_bf16(const void* A, const void* B, float* C, int M, int N, int T,
                         uint32_t* dev_words, void* stream) {
  if (M < 0 || N <= 0 || T < 0 || !C || !A || !B || !dev_words) return LMOE_ERR_INVALID_ARG;
  if (M % 8 || N % 16) return LMOE_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return LMOE_ERR_INVALID_ARG;
  if (M == 0) return LMOE_OK;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0)
    return cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * sizeof(float), st) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
  int32_t* seg = reinterpret_cast<int32_t*>(dev_words + 2);
  int rc = launch_rowmap(0, 0, nullptr, seg, T, st);  // writes seg = {0, T} and no map
  if (rc != LMOE_OK) return rc;
  GemmArgs g = gemm_defaults(dev_words, 1.0f);
  g.M = M;
  g.N = N;
  g.epi = EPI_F32;
  g.outf = C;
  g.ldf = N;
  g.groups = 1;
  g.kseg = seg;
  g.kfull = T;
  return launch_gemm(A, static_cast<uint64_t>(T), M, B, static_cast<uint64_t>(T), N, g, st);
}

size_t lmoe_packed_backward_bytes(const lmoe_dims* dims) {
  if (dims_supported(dims) != LMOE_OK || dims->expert_fp8) return 0;
  return bwd_packed_layout(*dims).total;
}

int lmoe_pack_backward_weights(const lmoe_dims* dims, const lmoe_weights* w, const void* packed,
                               void* packed_bwd, size_t bytes, void* stream) {
  const int rc0 = dims_supported(dims);
  if (rc0 != LMOE_OK) return rc0;
  const lmoe_dims D = *dims;
  if (D.expert_fp8) return LMOE_ERR_UNSUPPORTED;
  if (!w || !packed || !packed_bwd || !w->w_gate || !w->w_value || !w->w_edown ||
      !aligned16(packed) || !aligned16(packed_bwd))
    return LMOE_ERR_INVALID_ARG;
  const BwdPacked B = bwd_packed_layout(D);
  if (bytes < B.total) return LMOE_ERR_WORKSPACE_TOO_SMALL;
  using bf = __nv_bfloat16;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(packed_bwd);
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  const PackedLayout P = packed_layout(D);
  const int sw = shared_width(D), wz = D.L + sw, wc = D.L + 2 * sw, Ep = pad64(D.E);
  int rc = launch_pack_backward(D, *w, reinterpret_cast<bf*>(base + B.wgu_t),
                                reinterpret_cast<bf*>(base + B.wed_t), st);
  // dense weights: [W_up | W_sd] [d, L + sw] -> [L + sw, d]; W_r [E, L] -> [L, E padded];
  // [W_down ; shared gate/value] [L + 2 sw, d] -> [d, L + 2 sw]
  if (rc == LMOE_OK)
    rc = launch_transpose_rows(reinterpret_cast<const bf*>(pk + P.w2), wz, wz, D.d, D.d, D.d,
                               reinterpret_cast<bf*>(base + B.wout_t), st);
  if (rc == LMOE_OK)
    rc = launch_transpose_rows(reinterpret_cast<const bf*>(pk + P.wr), D.L, D.L, D.E, Ep, Ep,
                               reinterpret_cast<bf*>(base + B.wr_t), st);
  if (rc == LMOE_OK)
    rc = launch_transpose_rows(reinterpret_cast<const bf*>(pk + P.w1), D.d, D.d, wc, wc, wc,
                               reinterpret_cast<bf*>(base + B.wls_t), st);
  return rc;
}

size_t lmoe_routed_backward_workspace_bytes(const lmoe_dims* dims) {
  if (dims_supported(dims) != LMOE_OK || dims->expert_fp8) return 0;
  return bwd_layout(*dims).total;
}

int lmoe_routed_backward(const lmoe_dims* dims, const void* packed, const void* packed_bwd,
                         void* workspace, size_t ws_bytes, const float* dz, const void* pre,
                         float* dlat,
                         float* dgate, float* dgamma, float* dw_gu, float* dw_ed, void* bwd_ws,
                         size_t bwd_ws_bytes, void* stream_) {
  int rc = dims_supported(dims);
  if (rc != LMOE_OK) return rc;
  const lmoe_dims D = *dims;
  if (D.expert_fp8) return LMOE_ERR_UNSUPPORTED;
  if (!packed || !packed_bwd || !workspace || !dz || !dlat || !dgate || !dgamma || !dw_gu ||
      !dw_ed || !bwd_ws)
    return LMOE_ERR_INVALID_ARG;
  const void* ptrs[] = {packed, packed_bwd, workspace, dz, dlat, dgamma, dw_gu, dw_ed, bwd_ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LMOE_ERR_INVALID_ARG;
  RoutedBwd R{};
  R.D = D;
  R.W = workspace_layout(D);
  R.B = bwd_layout(D);
  if (ws_bytes < R.W.total_base || bwd_ws_bytes < R.B.total) return LMOE_ERR_WORKSPACE_TOO_SMALL;
  if (D.T == 0) return LMOE_OK;
  R.pk = static_cast<const uint8_t*>(packed);
  R.pb = static_cast<const uint8_t*>(packed_bwd);
  R.ws = static_cast<uint8_t*>(workspace);
  R.bw = static_cast<uint8_t*>(bwd_ws);
  R.P = packed_layout(D);
  R.PB = bwd_packed_layout(D);
  R.stream = static_cast<cudaStream_t>(stream_);
  if (pre && !aligned16(pre)) return LMOE_ERR_INVALID_ARG;
  R.pre = static_cast<const __nv_bfloat16*>(pre);
  if ((rc = routed_bwd_front(R, dz, dgate, dgamma)) != LMOE_OK) return rc;
  return routed_bwd_back(R, nullptr, dlat, nullptr, 0, dw_gu, dw_ed);
}

size_t lmoe_backward_workspace_bytes(const lmoe_dims* dims) {
  if (dims_supported(dims) != LMOE_OK || dims->expert_fp8) return 0;
  return layer_bwd_layout(*dims).total;
}

int lmoe_backward(const lmoe_dims* dims, const void* packed, const void* packed_bwd,
                  void* workspace, size_t ws_bytes, const void* x, const float* logits,
                  const void* dy, const void* pre, const void* pre_shared, float* dx,
                  float* dgamma, float* dw_in,
                  float* dw_router,
                  float* dw_gu, float* dw_ed, float* dw_out, void* bwd_ws, size_t bwd_ws_bytes,
                  void* stream_) {
  int rc = dims_supported(dims);
  if (rc != LMOE_OK) return rc;
  const lmoe_dims D = *dims;
  if (D.expert_fp8) return LMOE_ERR_UNSUPPORTED;
  if (!packed || !packed_bwd || !workspace || !x || !dy || !dx || !dgamma || !dw_in ||
      !dw_router || !dw_gu || !dw_ed || !dw_out || !bwd_ws)
    return LMOE_ERR_INVALID_ARG;
  const void* ptrs[] = {packed, packed_bwd, workspace, x, dy, dx, dgamma, dw_in, dw_router,
                        dw_gu, dw_ed, dw_out, bwd_ws};
  if ((pre && !aligned16(pre)) || (pre_shared && !aligned16(pre_shared)))
    return LMOE_ERR_INVALID_ARG;
  for (const void* p : ptrs)
    if (!aligned16(p)) return LMOE_ERR_INVALID_ARG;
  RoutedBwd R{};
  R.D = D;
  R.W = workspace_layout(D);
  R.B = bwd_layout(D);
  const LayerBwdLayout LB = layer_bwd_layout(D);
  if (ws_bytes < R.W.total_base || bwd_ws_bytes < LB.total) return LMOE_ERR_WORKSPACE_TOO_SMALL;
  if (D.T == 0) return LMOE_OK;
  using bf = __nv_bfloat16;
  R.pk = static_cast<const uint8_t*>(packed);
  R.pb = static_cast<const uint8_t*>(packed_bwd);
  R.ws = static_cast<uint8_t*>(workspace);
  R.bw = static_cast<uint8_t*>(bwd_ws);
  R.P = packed_layout(D);
  R.PB = bwd_packed_layout(D);
  R.stream = static_cast<cudaStream_t>(stream_);
  R.pre = static_cast<const __nv_bfloat16*>(pre);
  cudaStream_t stream = R.stream;
  const uint8_t* pk = R.pk;
  const uint8_t* pb = R.pb;
  uint8_t* ws = R.ws;
  uint8_t* bw = R.bw;
  const int T = D.T, L = D.L, E = D.E, d = D.d;
  const int sw = LB.sw, wc = LB.wc, wz = LB.wz, Ep = LB.Ep;
  uint32_t* err = reinterpret_cast<uint32_t*>(ws + R.W.err);
  const bf* xb = static_cast<const bf*>(x);
  const bf* dyb = static_cast<const bf*>(dy);
  const bf* lat = reinterpret_cast<const bf*>(ws + R.W.lat);
  const bf* zh = reinterpret_cast<const bf*>(ws + R.W.zh);
  const float* z = logits ? logits : reinterpret_cast<const float*>(ws + R.W.logits);
  float* dz = reinterpret_cast<float*>(bw + LB.dz);
  bf* dhs = reinterpret_cast<bf*>(bw + LB.dhs);
  float* dgate = reinterpret_cast<float*>(bw + LB.dgate);
  bf* dlogit = reinterpret_cast<bf*>(bw + LB.dlogit);
  float* dlat_r = reinterpret_cast<float*>(bw + LB.dlat_r);
  bf* dcat = reinterpret_cast<bf*>(bw + LB.dcat);
  bf* pre_s = reinterpret_cast<bf*>(bw + LB.pre_s);
  int32_t* seg1 = reinterpret_cast<int32_t*>(bw + LB.seg1);
  int32_t* rowmap_s = reinterpret_cast<int32_t*>(bw + LB.rowmap_s);
  // C[M, N] = A[M, Kd] . B[N, Kd]^T, fp32 or bf16 out
  auto dense = [&](const void* A, int M, int a_ld, const void* Bm, int N, int b_ld, int Kd,
                   int epi, void* out, int ld) {
    GemmArgs g = gemm_defaults(err, D.c);
    g.M = M;
    g.N = N;
    g.Kd = Kd;
    g.epi = epi;
    if (epi == EPI_F32) {
      g.outf = static_cast<float*>(out);
      g.ldf = ld;
    } else {
      g.out0 = static_cast<bf*>(out);
      g.ld0 = ld;
    }
    return launch_gemm(A, static_cast<uint64_t>(M), a_ld, Bm, static_cast<uint64_t>(N), b_ld, g,
                       stream);
  };
  // weight gradient dW[M, N] = A^T B over the T token rows of A [T, M] and B [T, N]
  auto wgrad = [&](const bf* Am, int M, int a_ld, const bf* Bm, int N, int b_ld, float* out,
                   const int32_t* row_map) {
    GemmArgs g = gemm_defaults(err, D.c);
    g.M = M;
    g.N = N;
    g.epi = EPI_F32;
    g.outf = out;
    g.ldf = N;
    g.groups = 1;
    g.kseg = seg1;
    g.kfull = T;  // the one group is every row of the operands
    g.row_map = row_map;
    return launch_gemm(Am, static_cast<uint64_t>(T), a_ld, Bm, static_cast<uint64_t>(T), b_ld, g,
                       stream);
  };
  // output rows of dw_in (shared gate/value rows de-interleaved), and the one-group range
  if ((rc = launch_rowmap(sw, L, rowmap_s, seg1, T, stream)) != LMOE_OK) return rc;
  // 1. [dz | dhs] = dy . [W_up | W_sd]  (dz fp32 for the RMSNorm backward, dhs bf16)
  if ((rc = dense(dyb, T, d, pb + R.PB.wout_t, L, d, d, EPI_F32, dz, L)) != LMOE_OK) return rc;
  if (sw > 0 && (rc = dense(dyb, T, d, pb + R.PB.wout_t + static_cast<size_t>(L) * d * 2, sw, d,
                            d, EPI_BF16, dhs, sw)) != LMOE_OK)
    return rc;
  // 2. routed branch, first half: dout, dgate, dgamma
  if ((rc = routed_bwd_front(R, dz, dgate, dgamma)) != LMOE_OK) return rc;
  // 3. router: dlogit, then its latent gradient dlat_r = dlogit . W_r
  if ((rc = launch_router_bwd(z, E, reinterpret_cast<const int32_t*>(ws + R.W.idx),
                              reinterpret_cast<const float*>(ws + R.W.gate), dgate, T, D.K,
                              dlogit, Ep, stream)) != LMOE_OK ||
      (rc = dense(dlogit, T, Ep, pb + R.PB.wr_t, L, Ep, Ep, EPI_F32, dlat_r, L)) != LMOE_OK)
    return rc;
  // 4. routed branch, second half: dlat = routed + router parts, bf16 into dcat[:, :L];
  // expert weight gradients
  if ((rc = routed_bwd_back(R, dlat_r, reinterpret_cast<float*>(bw + LB.dlat), dcat, wc, dw_gu,
                            dw_ed)) != LMOE_OK)
    return rc;
  // 5. shared experts: gate/value pre-activations (the forward's, or computed again), SiTU
  // backward into dcat[:, L:]
  if (sw > 0) {
    const bf* pre_sh = static_cast<const bf*>(pre_shared);
    if (!pre_sh) {
      if ((rc = dense(xb, T, d, pk + R.P.w1 + static_cast<size_t>(L) * d * 2, 2 * sw, d, d,
                      EPI_BF16, pre_s, 2 * sw)) != LMOE_OK)
        return rc;
      pre_sh = pre_s;
    }
    if ((rc = launch_situ_bwd(pre_sh, dhs, T, sw, D.c, dcat + L, wc, stream)) != LMOE_OK)
      return rc;
  }
  // 6. dx = [dlat | dgv_shared] . [W_down ; W_shared_gate/value]
  if ((rc = dense(dcat, T, wc, pb + R.PB.wls_t, d, wc, wc, EPI_F32, dx, d)) != LMOE_OK) return rc;
  // 7. dense weight gradients over the tokens: dw_out = dy^T [z | hs],
  // dw_router = dlogit^T lat, dw_in = [dlat | dgv_s]^T x
  if ((rc = wgrad(dyb, d, d, zh, wz, wz, dw_out, nullptr)) != LMOE_OK ||
      (rc = wgrad(dlogit, E, Ep, lat, L, L, dw_router, nullptr)) != LMOE_OK ||
      (rc = wgrad(dcat, wc, wc, xb, d, d, dw_in, rowmap_s)) != LMOE_OK)
    return rc;
  return LMOE_OK;
}

int lmoe_last_device_error(void* workspace) {
  if (!workspace) return LMOE_ERR_INVALID_ARG;
  uint32_t flag = 0;
  if (cudaMemcpy(&flag, workspace, sizeof flag, cudaMemcpyDeviceToHost) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (flag == 0) return LMOE_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(workspace, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (flag & (DEVERR_BAD_INDEX | DEVERR_NONFINITE)) return LMOE_ERR_INVALID_ARG;
  return LMOE_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"

// The argument checks of lmoe_forward for a batch of T > 0 tokens (LMOE_OK or the status
// lmoe_forward returns before it enqueues anything).
int lmoe::forward_args_check(const lmoe_dims* dims, const void* packed, const void* x,
                             const void* residual, const void* y, const void* workspace,
                             size_t ws_bytes, const lmoe_io* io) {
  int rc = dims_supported(dims);
  if (rc != LMOE_OK) return rc;
  const lmoe_dims D = *dims;
  lmoe_io opt{};
  opt.balance = 1;
  if (io) opt = *io;
  if (opt.phase < LMOE_PHASE_ALL || opt.phase > LMOE_PHASE_EXPERTS) return LMOE_ERR_INVALID_ARG;
  const bool front = opt.phase != LMOE_PHASE_EXPERTS;
  const bool back = opt.phase != LMOE_PHASE_ROUTER;
  if (opt.cand_out && (opt.phase != LMOE_PHASE_ROUTER || opt.cand_k < 1))
    return LMOE_ERR_INVALID_ARG;
  if (!packed || !workspace || (front && !x) || (back && !y)) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(packed) || !aligned16(workspace) || (front && !aligned16(x)) ||
      (back && !aligned16(y)) || (residual && !aligned16(residual)))
    return LMOE_ERR_INVALID_ARG;
  if (back && ((x && y == x) || (residual && y == residual))) return LMOE_ERR_INVALID_ARG;
  if (ws_bytes < workspace_layout(D).total_base) return LMOE_ERR_WORKSPACE_TOO_SMALL;
  if ((opt.tau_in && !aligned16(opt.tau_in)) || (opt.logits_in && !aligned16(opt.logits_in)))
    return LMOE_ERR_INVALID_ARG;
  if (opt.tau_ema && !(opt.ema_beta >= 0.0f && opt.ema_beta <= 1.0f)) return LMOE_ERR_INVALID_ARG;
  if (opt.save_pre && (D.expert_fp8 || !aligned16(opt.save_pre))) return LMOE_ERR_INVALID_ARG;
  if (opt.save_pre_shared && !aligned16(opt.save_pre_shared)) return LMOE_ERR_INVALID_ARG;
  if (opt.y_f32_out && !aligned16(opt.y_f32_out)) return LMOE_ERR_INVALID_ARG;
  if (opt.logit_bias && !aligned16(opt.logit_bias)) return LMOE_ERR_INVALID_ARG;
  return LMOE_OK;
}

extern "C" {

int lmoe_forward(const lmoe_dims* dims, const void* packed, const void* x, const void* residual,
                 void* y, void* workspace, size_t ws_bytes, lmoe_io* io, void* stream_) {
  if (io) io->kernel_launches = 0;
  int rc = dims_supported(dims);
  if (rc != LMOE_OK) return rc;
  const lmoe_dims D = *dims;
  lmoe_io opt{};
  opt.balance = 1;
  if (io) opt = *io;
  if (opt.phase < LMOE_PHASE_ALL || opt.phase > LMOE_PHASE_EXPERTS) return LMOE_ERR_INVALID_ARG;
  // front: latent/shared GEMM and router; back: thresholds through the output GEMM
  const bool front = opt.phase != LMOE_PHASE_EXPERTS;
  const bool back = opt.phase != LMOE_PHASE_ROUTER;
  if (opt.cand_out && (opt.phase != LMOE_PHASE_ROUTER || opt.cand_k < 1))
    return LMOE_ERR_INVALID_ARG;
  if (D.T == 0) {
    if (opt.cand_out)
      return launch_candidates(nullptr, 0, D.E, D.E, 1, opt.cand_k, opt.cand_out, D.E,
                               static_cast<cudaStream_t>(stream_));
    return LMOE_OK;
  }
  rc = forward_args_check(dims, packed, x, residual, y, workspace, ws_bytes, io);
  if (rc != LMOE_OK) return rc;
  const WorkspaceLayout W = workspace_layout(D);
  // Small whole-layer calls split the dense GEMMs' reductions when the workspace holds the
  // partials.  The two phases never do: a batch split across ranks then routes on logits
  // bit-identical to the whole batch's, whatever each part's size.
  const bool splitk =
      W.total > W.total_base && ws_bytes >= W.total && opt.phase == LMOE_PHASE_ALL;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  using bf = __nv_bfloat16;
  int launches = 0;
  // stage boundary: optional timing event; counts the kernels of the stage just finished
  StageRanges ranges;
  auto mark = [&](int stage_done_next, int kernels) -> bool {
    launches += kernels;
    ranges.enter(stage_done_next);
    if (!opt.stage_events) return true;
    cudaEvent_t ev = static_cast<cudaEvent_t>(opt.stage_events[stage_done_next]);
    return ev == nullptr || cudaEventRecord(ev, stream) == cudaSuccess;
  };
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  const PackedLayout P = packed_layout(D);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws + W.err);
  bf* lat = reinterpret_cast<bf*>(ws + W.lat);
  bf* zh = reinterpret_cast<bf*>(ws + W.zh);
  const int sw = shared_width(D);
  // the dense GEMMs' split-K scratch (one GEMM at a time, in stream order)
  auto dense_split = [&](GemmArgs& g) {
    if (!splitk) return;
    g.partial = reinterpret_cast<float*>(ws + W.splitk);
    g.partial_bytes = SPLITK_BYTES;
    g.extra_launches = &launches;
  };
  const int ldz = D.L + sw;
  const int T = D.T, TK = D.T * D.K;

  if (front && cudaMemsetAsync(err, 0, sizeof(uint32_t), stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (front && !mark(LMOE_STAGE_LATENT_SHARED, 0)) return LMOE_ERR_CUDA;

  int dev_sms = 0;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&dev_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  // Overlap: the shared experts (pure tensor work) run on an auxiliary stream on
  // `shared_ctas` SMs while the routed path (bandwidth-bound expert GEMMs) runs on the rest.
  const bool overlap = opt.aux_stream != nullptr && opt.aux_events[0] != nullptr &&
                       opt.aux_events[1] != nullptr && sw > 0 && T >= LMOE_OVERLAP_MIN_T;
  cudaStream_t aux = static_cast<cudaStream_t>(opt.aux_stream);
  int shared_ctas = 0, routed_ctas = 0;
  float* ys = nullptr;
  if (overlap) {
    shared_ctas = opt.shared_sms > 0 ? opt.shared_sms : dev_sms / 3;
    if (shared_ctas >= dev_sms) shared_ctas = dev_sms / 3;
    if (shared_ctas < 1) shared_ctas = 1;
    routed_ctas = dev_sms - shared_ctas;
    ys = reinterpret_cast<float*>(ws + W.ys);
  }

  if (!front) {
    // LMOE_PHASE_EXPERTS: the latent, shared activations and logits are in the workspace
  } else if (!overlap) {
    // 1. x . [W_down ; W_shared_gate/value]^T: latent (bf16) and SiTU(shared) into zh[:, L:]
    GemmArgs g = gemm_defaults(err, D.c);
    g.M = T;
    g.N = D.L + 2 * sw;
    g.Kd = D.d;
    g.epi = EPI_SPLIT;
    g.split = D.L;
    g.out0 = lat;
    g.ld0 = D.L;
    g.out1 = zh + D.L;
    g.ld1 = ldz;
    g.pre = static_cast<bf*>(opt.save_pre_shared);
    g.ldp = 2 * sw;
    g.inject_stall = inject_stall() ? 1 : 0;
    dense_split(g);
    rc = launch_gemm(x, T, D.d, pk + P.w1, static_cast<uint64_t>(g.N), D.d, g, stream);
    if (rc != LMOE_OK) return rc;
    launches += 1;
  } else {
    cudaEvent_t ev_fork = static_cast<cudaEvent_t>(opt.aux_events[0]);
    cudaEvent_t ev_join = static_cast<cudaEvent_t>(opt.aux_events[1]);
    if (cudaEventRecord(ev_fork, stream) != cudaSuccess ||
        cudaStreamWaitEvent(aux, ev_fork, 0) != cudaSuccess)
      return LMOE_ERR_CUDA;
    // aux 1: hs = SiTU(x . W_shared_gate/value^T) -> zh[:, L:]
    {
      GemmArgs g = gemm_defaults(err, D.c);
      g.M = T;
      g.N = 2 * sw;
      g.Kd = D.d;
      g.epi = EPI_SITU;
      g.out1 = zh + D.L;
      g.ld1 = ldz;
      g.pre = static_cast<bf*>(opt.save_pre_shared);
      g.ldp = 2 * sw;
      g.max_ctas = shared_ctas;
      rc = launch_gemm(x, T, D.d, pk + P.w1 + static_cast<size_t>(D.L) * D.d * 2,
                       static_cast<uint64_t>(2 * sw), D.d, g, aux);
      if (rc != LMOE_OK) return rc;
    }
    // aux 2: ys = hs . W_shared_down^T (fp32)
    {
      GemmArgs g = gemm_defaults(err, D.c);
      g.M = T;
      g.N = D.d;
      g.Kd = sw;
      g.epi = EPI_F32;
      g.outf = ys;
      g.ldf = D.d;
      g.max_ctas = shared_ctas;
      rc = launch_gemm(zh + D.L, T, ldz, pk + P.w2 + static_cast<size_t>(D.L) * 2,
                       static_cast<uint64_t>(D.d), ldz, g, aux);
      if (rc != LMOE_OK) return rc;
    }
    if (cudaEventRecord(ev_join, aux) != cudaSuccess) return LMOE_ERR_CUDA;
    // main 1: lat = x . W_down^T
    {
      GemmArgs g = gemm_defaults(err, D.c);
      g.M = T;
      g.N = D.L;
      g.Kd = D.d;
      g.epi = EPI_BF16;
      g.out0 = lat;
      g.ld0 = D.L;
      g.max_ctas = routed_ctas;
      g.inject_stall = inject_stall() ? 1 : 0;
      rc = launch_gemm(x, T, D.d, pk + P.w1, static_cast<uint64_t>(D.L), D.d, g, stream);
      if (rc != LMOE_OK) return rc;
    }
    launches += 3;
  }
  if (front && !mark(LMOE_STAGE_ROUTER, 0)) return LMOE_ERR_CUDA;
  // 2. router logits = lat . W_r^T (fp32), unless the caller supplies them
  const float* logits =
      opt.logits_in ? opt.logits_in : reinterpret_cast<const float*>(ws + W.logits);
  float* logits_t = reinterpret_cast<float*>(ws + W.logits_t);  // expert-major copy
  const bool solve_tau = !opt.tau_in && opt.balance;
  // the candidates of a router phase read the logits expert-major; in-batch thresholds read
  // the scores expert-major, which the scores kernel writes into the same buffer
  const bool want_t = opt.phase == LMOE_PHASE_ROUTER && opt.cand_out;
  if (front && !opt.logits_in) {
    GemmArgs g = gemm_defaults(err, D.c);
    g.M = T;
    g.N = D.E;
    g.Kd = D.L;
    g.epi = EPI_F32;
    g.outf = reinterpret_cast<float*>(ws + W.logits);
    g.ldf = D.E;
    g.col_bias = opt.logit_bias;
    g.max_ctas = routed_ctas;
    if (want_t) {
      g.outf_t = logits_t;
      g.ldt = T;
    }
    dense_split(g);
    rc = launch_gemm(lat, T, D.L, pk + P.wr, static_cast<uint64_t>(D.E), D.L, g, stream);
    if (rc != LMOE_OK) return rc;
    launches += 1;
  } else if (front && want_t) {
    rc = launch_transpose_f32(logits, T, D.E, logits_t, stream);
    if (rc != LMOE_OK) return rc;
    launches += 1;
  }
  // checked mode: the logits routed on (computed or given) must be finite
  if (front && check_finite()) {
    rc = launch_finite_check(logits, static_cast<int64_t>(T) * D.E, err, stream);
    if (rc != LMOE_OK) return rc;
    launches += 1;
  }
  auto copy = [&](void* dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, stream) == cudaSuccess;
  };
  if (!back) {
    // LMOE_PHASE_ROUTER ends here, with the candidates this batch contributes
    if (opt.cand_out) {
      rc = launch_candidates(logits_t, T, D.E, 1, T, opt.cand_k, opt.cand_out, D.E, stream);
      if (rc != LMOE_OK) return rc;
      launches += 1;
    }
    if (!mark(LMOE_STAGE_THRESHOLDS, 0)) return LMOE_ERR_CUDA;
    if (io) io->kernel_launches = launches;
    if (opt.logits_out && !copy(opt.logits_out, logits, static_cast<size_t>(T) * D.E * 4))
      return LMOE_ERR_CUDA;
    return LMOE_OK;
  }
  if (!mark(LMOE_STAGE_THRESHOLDS, 0)) return LMOE_ERR_CUDA;
  // 3. thresholds, on scores computed once for them and the selection
  const float* tau = opt.tau_in;
  const float* scores = reinterpret_cast<float*>(ws + W.scores);
  if (solve_tau) {
    rc = launch_scores(logits, T, D.E, reinterpret_cast<float*>(ws + W.scores), logits_t, stream);
    if (rc != LMOE_OK) return rc;
    launches += 1;
    float* t = reinterpret_cast<float*>(ws + W.tau);
    const int k = lmoe_fair_share_rank(T, D.K, D.E);
    rc = launch_thresholds(logits_t, T, D.E, 1, T, k, t, true, stream);
    if (rc != LMOE_OK) return rc;
    tau = t;
    launches += 1;
    if (opt.tau_ema) {
      // streaming thresholds: fold this batch's in, route against the result
      rc = launch_tau_ema(t, opt.tau_ema, D.E, opt.ema_beta, opt.ema_first ? 1 : 0, stream);
      if (rc != LMOE_OK) return rc;
      tau = opt.tau_ema;
      launches += 1;
    }
  }
  if (!mark(LMOE_STAGE_ROUTE, 0)) return LMOE_ERR_CUDA;
  // 4. top-K routing
  int32_t* idx = reinterpret_cast<int32_t*>(ws + W.idx);
  float* gate = reinterpret_cast<float*>(ws + W.gate);
  rc = solve_tau ? launch_route(scores, tau, T, D.E, D.K, idx, gate, nullptr, true, stream)
                  : launch_route(logits, tau, T, D.E, D.K, idx, gate, nullptr, false, stream);
  if (rc != LMOE_OK) return rc;
  if (!mark(LMOE_STAGE_DISPATCH, 1)) return LMOE_ERR_CUDA;
  // 5. dispatch into expert-contiguous segments
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + W.offsets);
  int32_t* ct_off = reinterpret_cast<int32_t*>(ws + W.ct_off);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + W.inv);
  int32_t* src_tok = reinterpret_cast<int32_t*>(ws + W.src_tok);
  // Chunk prefix sums: the batch's (which the backward reads), and a second one for the routed
  // GEMM that takes its own chunks -- the bf16 gate/value GEMM or the e4m3 down GEMM, never both
  const int tokn = grouped_tokn(T, D.K, D.E);
  const int tokn_gu = grouped_tokn_gate_up(T, D.K, D.E, D.expert_fp8 != 0);
  const int tokn_dn = grouped_tokn_down(T, D.K, D.E, D.expert_fp8 != 0);
  if (tokn_gu != tokn && tokn_dn != tokn) return LMOE_ERR_UNSUPPORTED;
  const int tokn2 = tokn_gu != tokn ? tokn_gu : tokn_dn;
  int32_t* ct_off2 = tokn2 != tokn ? reinterpret_cast<int32_t*>(ws + W.ct_off2) : nullptr;
  int32_t* ct_off_gu = tokn_gu != tokn ? ct_off2 : ct_off;
  int32_t* ct_off_dn = tokn_dn != tokn ? ct_off2 : ct_off;
  rc = launch_dispatch(idx, T, D.E, D.K, reinterpret_cast<uint32_t*>(ws + W.masks),
                       reinterpret_cast<uint32_t*>(ws + W.base), offsets, ct_off, tokn, ct_off2,
                       tokn2, inv, src_tok, opt.counts_out, err, stream);
  if (rc != LMOE_OK) return rc;
  if (opt.load_stats) {
    rc = launch_load_stats(nullptr, offsets, D.E, opt.load_stats, stream);
    if (rc != LMOE_OK) return rc;
    launches += 1;
  }
  if (!mark(LMOE_STAGE_EXPERT_GATE_UP, 3)) return LMOE_ERR_CUDA;
  // 6. routed gate/value GEMM with SiTU-GLU: h = SiTU(lat[src_tok] . W_gu[e]^T) per expert,
  //    the latent rows gathered inside the GEMM
  bf* h = reinterpret_cast<bf*>(ws + W.h);
  const bool fp8 = D.expert_fp8 != 0;
  {
    GroupedArgs g{};
    g.E = D.E;
    g.M_w = 2 * D.I;
    g.Kd = D.L;
    g.seg_off = offsets;
    g.ct_off = ct_off_gu;
    g.gather = src_tok;
    g.x = lat;
    g.ldx = D.L;
    const void* xop = lat;
    if (fp8) {
      // e4m3 latent rows (one scale per token), gathered like the bf16 rows
      uint8_t* lat8 = ws + W.lat8;
      float* slat = reinterpret_cast<float*>(ws + W.slat);
      rc = launch_quantize_rows(lat, T, D.L, D.L, lat8, D.L, slat, stream);
      if (rc != LMOE_OK) return rc;
      launches += 1;
      g.fp8 = 1;
      g.x = reinterpret_cast<const bf*>(lat8);
      g.w_scale = reinterpret_cast<const float*>(pk + P.sgu);
      g.x_scale = slat;
      xop = lat8;
    }
    g.epi = EPI_SITU;
    g.out = h;
    g.ldo = D.I;
    g.pre = static_cast<bf*>(opt.save_pre);
    g.ldp = 2 * D.I;
    g.c = D.c;
    g.err = err;
    g.timeout_ns = wait_limit_ns();
    g.max_ctas = routed_ctas;
    g.mean_tokens = static_cast<int>(static_cast<int64_t>(TK) / D.E);
    g.tokn = tokn_gu;
    rc = launch_grouped_gemm(pk + P.wgu, xop, static_cast<uint64_t>(T), D.L, g, stream);
    if (rc != LMOE_OK) return rc;
  }
  if (!mark(LMOE_STAGE_EXPERT_DOWN, 1)) return LMOE_ERR_CUDA;
  // 7. routed down GEMM: o = h . W_ed[e]^T per expert
  bf* o = reinterpret_cast<bf*>(ws + W.o);
  {
    GroupedArgs g{};
    g.E = D.E;
    g.M_w = D.L;
    g.Kd = D.I;
    g.seg_off = offsets;
    g.ct_off = ct_off_dn;
    g.epi = EPI_BF16;
    g.out = o;
    g.ldo = D.L;
    g.c = D.c;
    g.err = err;
    g.timeout_ns = wait_limit_ns();
    g.max_ctas = routed_ctas;
    g.mean_tokens = static_cast<int>(static_cast<int64_t>(TK) / D.E);
    g.tokn = tokn_dn;
    const void* xop = h;
    if (fp8) {
      // e4m3 SiTU outputs, one scale per (token, expert) row
      uint8_t* h8 = ws + W.h8;
      float* sh = reinterpret_cast<float*>(ws + W.sh);
      rc = launch_quantize_rows(h, TK, D.I, D.I, h8, D.I, sh, stream);
      if (rc != LMOE_OK) return rc;
      launches += 1;
      g.fp8 = 1;
      g.w_scale = reinterpret_cast<const float*>(pk + P.sed);
      g.x_scale = sh;
      xop = h8;
    }
    rc = launch_grouped_gemm(pk + P.wed, xop, static_cast<uint64_t>(TK), D.I, g, stream);
    if (rc != LMOE_OK) return rc;
  }
  if (!mark(LMOE_STAGE_COMBINE, 1)) return LMOE_ERR_CUDA;
  // 8. gate-weighted combine + RMSNorm -> zh[:, :L]
  rc = launch_combine(o, gate, inv, reinterpret_cast<const float*>(pk + P.gamma), T, D.K, D.L,
                      D.eps, zh, ldz, err, wait_limit_ns(), stream);
  if (rc != LMOE_OK) return rc;
  if (!mark(LMOE_STAGE_OUTPUT, 1)) return LMOE_ERR_CUDA;
  // 9. y = residual + [z | hs] . [W_up | W_sd]^T   (overlap: y = residual + z . W_up^T + ys)
  {
    GemmArgs g = gemm_defaults(err, D.c);
    g.M = T;
    g.N = D.d;
    g.epi = EPI_RESID;
    g.out0 = static_cast<bf*>(y);
    g.ld0 = D.d;
    g.resid = static_cast<const bf*>(residual);
    g.ldr = D.d;
    g.outf = opt.y_f32_out;
    g.ldf = D.d;
    if (!overlap) {
      g.Kd = ldz;
      dense_split(g);
      rc = launch_gemm(zh, T, ldz, pk + P.w2, static_cast<uint64_t>(D.d), ldz, g, stream);
    } else {
      if (cudaStreamWaitEvent(stream, static_cast<cudaEvent_t>(opt.aux_events[1]), 0) !=
          cudaSuccess)
        return LMOE_ERR_CUDA;
      g.Kd = D.L;
      g.addf = ys;
      g.lda = D.d;
      rc = launch_gemm(zh, T, ldz, pk + P.w2, static_cast<uint64_t>(D.d), ldz, g, stream);
    }
    if (rc != LMOE_OK) return rc;
  }
  if (!mark(LMOE_NUM_STAGES, 1)) return LMOE_ERR_CUDA;
  if (io) io->kernel_launches = launches;
  // debug outputs
  if (opt.logits_out && !copy(opt.logits_out, logits, static_cast<size_t>(T) * D.E * 4))
    return LMOE_ERR_CUDA;
  if (opt.tau_out) {
    const bool ok = tau ? copy(opt.tau_out, tau, static_cast<size_t>(D.E) * 4)
                        : cudaMemsetAsync(opt.tau_out, 0, static_cast<size_t>(D.E) * 4,
                                          stream) == cudaSuccess;
    if (!ok) return LMOE_ERR_CUDA;
  }
  if (opt.idx_out && !copy(opt.idx_out, idx, static_cast<size_t>(TK) * 4)) return LMOE_ERR_CUDA;
  if (opt.gate_out && !copy(opt.gate_out, gate, static_cast<size_t>(TK) * 4))
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

}  // extern "C"
