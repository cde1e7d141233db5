// libvla C ABI: handle life cycle, argument validation, weight repacking,
// the per-handle time-conditioning table, split-K planning and the solver
// loop (captured once per shape/pointer set into a CUDA graph and replayed).
//
// The call structure follows "vla.cpp: A Unified Inference Runtime for
// Vision-Language-Action Models": the prefix K/V cache is built once per
// observation (§III-B Eq. (2)) and reused by all S Euler steps of the action
// expert (§III-A Eq. (1)); for unchanged shapes the graph and buffers persist
// across calls (§III-B, latency model Eq. (3)).
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <new>
#include <vector>

#include "vla_common.cuh"

static thread_local char g_last_error[256] = "";

namespace {

struct GraphEntry {
  int B, P;
  const uint32_t* pmask;
  const void* kc;
  const void* vc;
  const float* noise;
  float* actions;
  float* tap;
  cudaGraphExec_t exec;
  uint64_t last_use;
};

constexpr int kMaxGraphs = 8;

struct GemmPlan {
  int splits = 1;
  int kb_per_split = 1;
  int BN = 16;
  int tiles_n = 1;
  int tiles_t = 1;
  int stages = 4;
};

int cdiv(int a, int b) { return (a + b - 1) / b; }

int round_up(int a, int b) { return cdiv(a, b) * b; }

}  // namespace

void vla_set_last_error(const char* where, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
}

struct vla_expert {
  vla_expert_config cfg{};
  int S = 0;
  bool w2a8 = false;
  bool f32 = false;
  bool use_tc = false;
  int num_sms = 0;
  size_t es = 2;
  int qdim = 0, kvdim = 0, qkvdim = 0, Kmax = 0, Hp = 0;
  // handle-owned weights
  void* wkv_pre = nullptr;  // [L*2*kvdim][d_vlm]: per layer K rows then V rows
  void* wqkv = nullptr;     // [L][qkvdim][D]  (W2A8: packed [L][qkvdim][D/4])
  void* wo = nullptr;       // [L][D][qdim]
  void* wup = nullptr;      // [L][F][D]
  void* wdown = nullptr;    // [L][D][F]
  float* beta = nullptr;    // [L][6] per-tensor scales (W2A8, CUDA-core path)
  float* beta_rows = nullptr;  // [L][qkvdim + D + F + D] per-output-row scales (W2A8)
  int beta_stride = 0, beta_group = 0;
  bool tpre = false;             // ternary prefix maps (W2A8 prefix build)
  float* beta_pre_rows = nullptr;  // [L][2 kvdim] their per-row scales
  void* zcodes = nullptr;          // Eq. (4) codes of the prefix rows (bf16 carriers)
  float* zalpha = nullptr;
  float* win = nullptr;     // [D][d_a]
  float* wout = nullptr;    // [d_a][D]
  float* modtab = nullptr;  // [S][L][4][D]
  float* modf = nullptr;    // [S][2][D]
  // workspace for max_batch x H tokens
  float* h = nullptr;
  void* act = nullptr;
  int8_t* codes = nullptr;
  float* alpha = nullptr;
  float* part = nullptr;
  size_t part_elems = 0;
  void* q = nullptr;
  void* ks = nullptr;
  void* vs = nullptr;
  float* opart = nullptr;
  float* ml = nullptr;
  int attn_chunk = 0;
  // fused tensor-core path (bf16): row sums of squares, tcgen05 attention partials
  bool fused = false;
  float* ss1 = nullptr;
  float* ss2 = nullptr;
  size_t ss_elems = 0;
  float* aopart = nullptr;
  float2* aml = nullptr;
  void* gbuf = nullptr;  // [T][F] bf16 GeLU output (separate from act: the up GEMM may read act)
  float* f32buf = nullptr;  // W2A8: fp32 attention / GeLU outputs [T][max(qdim, F)] awaiting quantisation
  unsigned long long* tl = nullptr;  // event trace buffer (VLA_TIMELINE builds)
  float* xpart = nullptr;  // split-K partial tiles exchanged through L2
  float* xss = nullptr;    // per-rank sums of squares exchanged through L2
  bf16* xo = nullptr;      // attention partial outputs exchanged through L2
  float2* xml = nullptr;   // and their row maxima and sums
  size_t xpart_elems = 0, xss_elems = 0;
  int* d_status = nullptr;
  int* h_abort = nullptr;
  int* d_abort = nullptr;
  CUtensorMap tm_wkv, tm_wqkv, tm_wo, tm_wup, tm_wdown;
  cudaStream_t cap_stream = nullptr;
  std::vector<GraphEntry> graphs;
  uint64_t tick = 0;
  // selected FFN neurons: effective MLP width and the compact weight copies
  int F_eff = 0;
  void* wup_full = nullptr;
  void* wdown_full = nullptr;
  void* wup_sel = nullptr;
  void* wdown_sel = nullptr;
  // request options of the call being enqueued (prefix mask) and the buffer
  // for in-library noise
  const uint32_t* pmask = nullptr;
  int pmw = 0;
  float* noise_buf = nullptr;
  // persistent whole-solve kernel for few tokens (k_solver_persist.cu)
  bool persist_ok = false;
  int persist_T = 0;         // tokens its buffers hold
  float* cqkv = nullptr;     // [S][L][qkvdim]  W_qkv beta_a per (step, layer)
  float* cup = nullptr;      // [S][L][F]       W_up beta_m
  // factored modulated norm of the many-token linears: (1 + gamma) h in bf16
  bf16* xt = nullptr;        // [max T][D]
  float* p_accq = nullptr;
  float* p_accu = nullptr;
  float* p_rms = nullptr;
  float* p_opart = nullptr;
  float2* p_oml = nullptr;
  unsigned* p_bar = nullptr;
  size_t p_units = 0;
  // diagnostic tap of one W2A8 solver step (vla_expert_set_w2a8_tap)
  void* tap = nullptr;
  size_t tap_cap = 0;
  int tap_step = -1;
  // request buffers (vla_policy_step_host), allocated on first use
  void* req_z = nullptr;
  void* req_kc = nullptr;
  void* req_vc = nullptr;
  float* req_noise = nullptr;
  float* req_act = nullptr;
};

namespace {

// Layer l attends to the cached prefix keys only (a cross-attention layer of
// the alternating joint / cross design) when cross_every > 0 and l mod
// cross_every == cross_every - 1.
bool is_cross(const vla_expert_config& c, int l) {
  return c.cross_every > 0 && l % c.cross_every == c.cross_every - 1;
}

// tau_{k+1} - tau_k of the handle's schedule: 1/S, or -1/S for the reverse
// (1 -> 0) convention, whose velocity sign change enters Eq. (1) here.
float step_dt(const vla_expert* h, int k) {
  const double d = (double)(k + 1) / h->S - (double)k / h->S;
  return (float)(h->cfg.schedule == VLA_SCHEDULE_REVERSE ? -d : d);
}

vla_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return VLA_OK;
  vla_set_last_error("CUDA", e);
  if (e == cudaErrorMemoryAllocation) return VLA_ERR_OOM;
  return VLA_ERR_CUDA;
}

#define VLA_ST(expr)              \
  do {                            \
    const vla_status _s = (expr); \
    if (_s != VLA_OK) return _s;  \
  } while (0)

#define VLA_CK(expr)                                   \
  do {                                                 \
    cudaError_t _e = (expr);                           \
    if (_e != cudaSuccess) {                           \
      vla_set_last_error(#expr, _e);                   \
      return _e == cudaErrorMemoryAllocation ? VLA_ERR_OOM : VLA_ERR_CUDA; \
    }                                                  \
  } while (0)

template <typename T>
vla_status dalloc(T** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc((void**)p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return VLA_ERR_OOM;
  }
  return VLA_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

GemmPlan plan_gemm(const vla_expert* h, int N, int K, int T) {
  GemmPlan p;
  if (h->use_tc && !h->w2a8) {
    p.BN = T >= 256 ? 256 : round_up(T < 16 ? 16 : T, 16);
    p.tiles_n = cdiv(N, 128);
    p.tiles_t = cdiv(T, p.BN);
    const int num_kb = K / 64;
    const int tiles = p.tiles_n * p.tiles_t;
    int s = h->num_sms / tiles;
    if (s < 1) s = 1;
    if (s > num_kb) s = num_kb;
    p.kb_per_split = cdiv(num_kb, s);
    p.splits = cdiv(num_kb, p.kb_per_split);
    const int stage = 128 * 128 + p.BN * 128;
    int st = (220 * 1024) / stage;
    if (st > 8) st = 8;
    if (st > p.kb_per_split) st = p.kb_per_split < 2 ? 2 : p.kb_per_split;
    p.stages = st;
  } else {
    const int tiles = cdiv(T, 64) * cdiv(N, 64);
    const int align = h->w2a8 ? 64 : 32;
    int s = h->num_sms / tiles;
    if (s < 1) s = 1;
    if (s > K / align) s = K / align > 0 ? K / align : 1;
    p.splits = simt_effective_splits(K, s, align);
  }
  return p;
}

void gemm_dims(const vla_expert* h, int which, int* N, int* K) {
  const int D = h->cfg.width, F = h->F_eff;
  switch (which) {
    case 0: *N = h->qkvdim; *K = D; break;
    case 1: *N = D; *K = h->qdim; break;
    case 2: *N = F; *K = D; break;
    default: *N = D; *K = F; break;
  }
}

ExpertDims make_dims(const vla_expert* h, int B, int P) {
  ExpertDims d;
  const vla_expert_config& c = h->cfg;
  d.L = c.n_layers; d.D = c.width; d.F = h->F_eff; d.n_q = c.n_q_heads; d.n_kv = c.n_kv_heads;
  d.d_h = c.head_dim; d.d_a = c.action_dim; d.H = c.horizon; d.B = B; d.P = P; d.S = h->S; d.d_t = c.time_dim;
  d.eps = c.rms_eps; d.qdim = h->qdim; d.kvdim = h->kvdim; d.qkvdim = h->qkvdim;
  d.f32 = h->f32 ? 1 : 0;
  d.w2a8 = h->w2a8 ? 1 : 0;
  d.P8 = round_up(P, 8);
  d.Hp = h->Hp;
  return d;
}

StepBufs make_bufs(const vla_expert* h, int P) {
  StepBufs b;
  b.win = h->win; b.wout = h->wout; b.modtab = h->modtab; b.modf = h->modf; b.beta = h->beta;
  b.h = h->h; b.act = h->act; b.codes = h->codes; b.alpha = h->alpha; b.part = h->part;
  b.q = h->q; b.ks = h->ks; b.vs = h->vs; b.opart = h->opart; b.ml = h->ml;
  b.attn_chunk = h->attn_chunk;
  b.n_chunks = cdiv(P + h->cfg.horizon, h->attn_chunk);
  b.pmask = h->pmask;
  b.pmw = h->pmw;
  return b;
}

cudaError_t run_linear(vla_expert* h, int which, int layer, int T, const GemmPlan& p, const CUtensorMap* tmX,
                       cudaStream_t st) {
  int N, K;
  gemm_dims(h, which, &N, &K);
  const void* wbase = which == 0 ? h->wqkv : which == 1 ? h->wo : which == 2 ? h->wup : h->wdown;
  const size_t sstride = (size_t)T * N;
  if (h->w2a8) {
    const uint8_t* q = (const uint8_t*)wbase + (size_t)layer * N * (K / 4);
    return launch_ternary_simt(h->codes, K, q, T, N, K, p.splits, h->part, sstride, N, st);
  }
  if (!h->use_tc) {
    const void* W = (const char*)wbase + (size_t)layer * N * K * h->es;
    return launch_gemm_simt(!h->f32, h->act, K, !h->f32, W, K, T, N, K, p.splits, h->part, sstride, N, nullptr,
                            st);
  }
  const CUtensorMap* tmW = which == 0 ? &h->tm_wqkv : which == 1 ? &h->tm_wo : which == 2 ? &h->tm_wup : &h->tm_wdown;
  TcGemmArgs a{};
  a.N = N; a.T = T; a.a_row0 = layer * N; a.num_kb = K / 64; a.kb_per_split = p.kb_per_split; a.BN = p.BN;
  a.stages = p.stages; a.out = h->part; a.split_stride = sstride; a.ldo = N; a.mode = 0; a.status = h->d_status;
  return launch_gemm_tc(tmW, tmX, a, p.tiles_n, p.tiles_t, p.splits, st);
}

vla_status enqueue_denoise(vla_expert* h, const void* kc, const void* vc, int B, int P, const float* noise,
                           float* actions, float* tap, cudaStream_t st) {
  const vla_expert_config& c = h->cfg;
  const ExpertDims d = make_dims(h, B, P);
  const StepBufs sb = make_bufs(h, P);
  const int T = B * c.horizon;
  GemmPlan pl[4];
  for (int w = 0; w < 4; ++w) {
    int N, K;
    gemm_dims(h, w, &N, &K);
    pl[w] = plan_gemm(h, N, K, T);
  }
  CUtensorMap tmX[3];  // activations [T][K] for K = D, qdim, F
  if (h->use_tc && !h->w2a8) {
    const int ks[3] = {c.width, h->qdim, h->F_eff};
    for (int i = 0; i < 3; ++i)
      if (tc_encode_2d_bf16(&tmX[i], h->act, ks[i], T, 64, pl[0].BN) != 0) return VLA_ERR_CUDA;
  }
  const CUtensorMap* xmap[4] = {&tmX[0], &tmX[1], &tmX[0], &tmX[2]};
  const DevCtl ctl{h->d_status, h->d_abort};
  for (int k = 0; k < h->S; ++k) {
    const float* x_in = k == 0 ? noise : actions;
    const float dt = step_dt(h, k);
    VLA_CK(launch_embed_norm(d, sb, k, x_in, ctl, st));
    for (int l = 0; l < c.n_layers; ++l) {
      VLA_CK(run_linear(h, 0, l, T, pl[0], xmap[0], st));
      VLA_CK(launch_reduce_qkv(d, sb, l, pl[0].splits, st));
      StepBufs sbl = sb;
      sbl.no_suffix = is_cross(c, l) ? 1 : 0;
      VLA_CK(launch_attention(d, sbl, l, kc, vc, st));
      VLA_CK(run_linear(h, 1, l, T, pl[1], xmap[1], st));
      VLA_CK(launch_reduce_norm(d, sb, k, l, 3, l, 1, pl[1].splits, st));
      VLA_CK(run_linear(h, 2, l, T, pl[2], xmap[2], st));
      VLA_CK(launch_reduce_gelu(d, sb, l, pl[2].splits, st));
      VLA_CK(run_linear(h, 3, l, T, pl[3], xmap[3], st));
      if (l + 1 < c.n_layers)
        VLA_CK(launch_reduce_norm(d, sb, k, l, 5, l + 1, 0, pl[3].splits, st));
      else
        VLA_CK(launch_head(d, sb, k, pl[3].splits, dt, x_in, actions, tap, st));
    }
  }
  return VLA_OK;
}

struct LinPlan {
  int C = 1, KS = 64, BN = 16, tiles_n = 1, tiles_t = 1, stages = 1, bmode = 0;
  int amode = 0;      // packed ternary weights: 1 (code ring) or 2 (every k-block's codes resident)
  bool wide = false;  // persistent many-token kernel (k_linear_wide.cu)
  int grid = 0;       // its CTA count
};

// Many-token plan: the persistent kernel with 128 x BN tiles, BN a multiple
// of 16 in [64, 256] chosen to minimise waves x (BN + 64) (the tile's token
// columns plus a fixed per-tile cost of about 64 columns, measured: four
// waves of 176 took longer than three of 256 for 512 prefix tokens); e.g.
// 3200 action tokens take QKV tiles of 224 (two waves) instead of 256.  Used when even 128-token tiles give a
// wave of work for every SM (or always, with VLA_FLAG_LINEAR_WIDE); never for
// packed ternary weights.
LinPlan plan_wide(int num_sms, int N, int K, int T) {
  LinPlan p;
  const int tn = N / 128;
  long best = -1;
  for (int bn = 256; bn >= 64; bn -= 16) {
    const long cost = (long)cdiv(tn * cdiv(T, bn), num_sms) * (bn + 64);
    if (best < 0 || cost < best) {
      best = cost;
      p.BN = bn;
    }
  }
  p.wide = true;
  p.C = 1;
  p.KS = K;
  p.tiles_n = tn;
  p.tiles_t = cdiv(T, p.BN);
  p.grid = p.tiles_n * p.tiles_t < num_sms ? p.tiles_n * p.tiles_t : num_sms;
  p.bmode = 0;
  p.stages = 4;
  return p;
}

bool wide_applies(unsigned flags, int num_sms, int N, int K, int T) {
  if ((flags & VLA_FLAG_LINEAR_SPLIT) || N % 128 || K % 64) return false;
  if (flags & VLA_FLAG_LINEAR_WIDE) return true;
  return (N / 128) * cdiv(T, 128) >= num_sms;
}

// Cluster split-K plan: the smallest power-of-two cluster (<= 16) that puts
// about one CTA on every SM, with the modulated-norm prologue fused when the
// CTA's B slice fits in shared memory.  Packed ternary weights: clusters of
// at most 8 and a ring of at most 90 KB, so that two CTAs (and the next
// kernel's early CTAs) fit on an SM and every grid runs as one wave (with
// 160 KB rings and clusters of 16 the batch-1 W2A8 O, up and down
// projections ran as two waves each; measured per solve: 16.45 -> 12.02 ms
// at B = 1, 23.48 -> 16.62 ms at B = 16; a 110 KB ring gave 12.16 / 16.93).
LinPlan plan_linear_sms(int num_sms, int N, int K, int T, bool want_norm, bool packed) {
  LinPlan p;
  p.BN = T >= 256 ? 256 : round_up(T < 16 ? 16 : T, 16);
  p.tiles_n = cdiv(N, 128);
  p.tiles_t = cdiv(T, p.BN);
  const int tiles = p.tiles_n * p.tiles_t;
  p.C = 1;
  const int cmax = packed ? 8 : 16;
  while (p.C < cmax && tiles * p.C < num_sms && K % (p.C * 2 * 64) == 0) p.C *= 2;
  p.KS = K / p.C;
  const int nkb = p.KS / 64;
  const int b_tile = p.BN * 128;
  const int b_res = nkb * b_tile;
  // the in-GEMM norm prologue maps a fixed 8-column chunk to each thread:
  // KS / 8 must divide 128
  const int kcs = p.KS / 8;
  p.bmode = (want_norm && b_res <= 96 * 1024 && kcs <= 128 && 128 % kcs == 0) ? 1 : 0;
  // packed codes: all of the CTA's k-blocks at once when they are few
  // (loaded together before the grid-dependency wait; the decode is then
  // paced by the decoders and the MMAs), else a ring beside the decoded tiles
  p.amode = packed ? (nkb <= 16 ? 2 : 1) : 0;
  const int resident = p.amode == 2 ? nkb * 128 * 16 : 0;
  const int budget = (packed ? 90 * 1024 : 200 * 1024) - (p.bmode ? b_res : 0) - resident;
  const int per_stage = 128 * 128 + (p.bmode ? 0 : b_tile) + (p.amode == 1 ? 128 * 16 : 0);
  int st = budget / per_stage;
  if (st > 8) st = 8;
  if (st > nkb) st = nkb;
  if (st < 1) st = 1;
  p.stages = st;
  return p;
}

LinPlan plan_linear(const vla_expert* h, int N, int K, int T, bool want_norm) {
  if (!h->w2a8 && wide_applies(h->cfg.flags, h->num_sms, N, K, T)) return plan_wide(h->num_sms, N, K, T);
  return plan_linear_sms(h->num_sms, N, K, T, want_norm && !h->w2a8, h->w2a8);
}

// The bf16 solver folds its modulated norms into the linears (see
// enqueue_denoise_fused) whenever the handle holds the W beta tables for its
// MLP width.
bool factored_norm(const vla_expert* h) { return h->xt && h->F_eff == h->cfg.mlp_width; }

// One linear layer on the kernel its plan names.
cudaError_t run_lin(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmH, const LinArgs& a,
                    const LinPlan& p, cudaStream_t st) {
  if (p.wide) return launch_linear_wide(tmA, tmB, a, p.grid, st);
  return launch_linear(tmA, tmB, tmH, a, p.tiles_n, p.tiles_t, p.C, st);
}

LinArgs lin_args(const vla_expert* h, const LinPlan& p, int N, int T, int layer) {
  LinArgs a{};
  a.N = N; a.T = T; a.a_row0 = layer * N; a.KS = p.KS; a.BN = p.BN; a.stages = p.stages; a.bmode = p.bmode;
  a.eps = h->cfg.rms_eps; a.D = h->cfg.width; a.status = h->d_status;
  a.H = h->cfg.horizon; a.n_q = h->cfg.n_q_heads; a.n_kv = h->cfg.n_kv_heads; a.d_h = h->cfg.head_dim;
  a.qdim = h->qdim; a.kvdim = h->kvdim; a.Hp = h->Hp;
  a.xpart = h->xpart; a.xss = h->xss;
  a.layer = layer;
  if (h->w2a8) {
    a.amode = p.amode; a.w2a8 = 1; a.alpha = h->alpha; a.wbeta = h->beta_rows; a.beta_stride = h->beta_stride;
  }
  return a;
}

// Attention cluster: cs - 1 ranks share the prefix keys (at most 128 each),
// the last rank takes the action keys.
int attn_cluster(int P) { return P <= 7 * 128 ? 8 : 16; }
int attn_kc(int P, int cs) {
  const int kc = round_up(cdiv(P, cs - 1), 16);
  return kc < 16 ? 16 : kc;
}

// Diagnostic W2A8 tap: for every layer of the tapped step, 22 tensors in this
// order, each starting on a 256-byte boundary (the layout vla.h documents).
constexpr int kTapTensors = 22;
void tap_sizes(const vla_expert* h, int B, size_t sz[kTapTensors]) {
  const vla_expert_config& c = h->cfg;
  const size_t T = (size_t)B * c.horizon, D = c.width, F = c.mlp_width, Q = h->qdim;
  const size_t v[kTapTensors] = {
      T * D * 4, T * D * 4, T * D * 2, T * 4, T * h->qkvdim * 4,                        // h_in u_a c_a al_a acc_qkv
      (size_t)B * c.n_q_heads * c.horizon * c.head_dim * 2,                             // q
      (size_t)B * c.n_kv_heads * c.horizon * c.head_dim * 2,                            // k_s
      (size_t)B * c.n_kv_heads * c.head_dim * h->Hp * 2,                                // v_s^T
      T * Q * 4, T * Q * 2, T * 4, T * D * 4, T * D * 4,                                // o32 c_o al_o acc_o h_mid
      T * D * 4, T * D * 2, T * 4, T * F * 4, T * F * 4, T * F * 2, T * 4, T * D * 4,   // u_m c_m al_m acc_up g32 c_d al_d acc_d
      T * D * 4};                                                                      // h_out
  for (int i = 0; i < kTapTensors; ++i) sz[i] = v[i];
}
size_t tap_pad(size_t b) { return (b + 255) / 256 * 256; }
size_t tap_layer_bytes(const vla_expert* h, int B) {
  size_t sz[kTapTensors], tot = 0;
  tap_sizes(h, B, sz);
  for (size_t x : sz) tot += tap_pad(x);
  return tot;
}
// Device address of tensor `i` of layer `l` in the tap.
char* tap_at(const vla_expert* h, int B, int l, int i) {
  size_t sz[kTapTensors], off = tap_layer_bytes(h, B) * (size_t)l;
  tap_sizes(h, B, sz);
  for (int j = 0; j < i; ++j) off += tap_pad(sz[j]);
  return (char*)h->tap + off;
}

bool fused_supported(const vla_expert_config& c, bool f32, bool w2a8, bool use_tc) {
  if (f32 || !use_tc) return false;
  (void)w2a8;
  if (c.head_dim % 64 || c.head_dim > 256 || c.width % 128 || c.horizon > 128) return false;
  if (c.max_prefix > 15 * 128) return false;
  if (!w2a8 && c.width / 128 > 16) return false;  // sums-of-squares slots read by the norm prologue
  const int cs = attn_cluster(c.max_prefix);
  if ((c.head_dim / cs) % 8) return false;
  const int kc = attn_kc(c.max_prefix, cs);
  const int kmax = kc > round_up(c.horizon, 16) ? kc : round_up(c.horizon, 16);
  return attn_tc_smem_bytes(c.head_dim, kmax) <= 227 * 1024;
}

// Attention for one solve: the kernel form, its arguments and tensor maps.
// The streaming kernel (one CTA per query tile, all keys; head sizes 64, 128
// and 256) is used when the query tiles alone occupy a fifth of the SMs;
// otherwise the clustered kernel spreads each tile's keys over a cluster.
// VLA_FLAG_ATTN_SPLIT / VLA_FLAG_ATTN_STREAM force one form (the streaming
// one only where it applies).
struct AttnPlan {
  bool stream;
  AttnArgs aa;
  CUtensorMap tmQ, tmK, tmVt, tmKs, tmVs;
};

vla_status plan_attention(const vla_expert* h, int B, int P, const void* kc, const void* vc, void* o, float* o32,
                          AttnPlan* ap) {
  const vla_expert_config& c = h->cfg;
  const int dh = c.head_dim, nkv = c.n_kv_heads, L = c.n_layers, P8 = round_up(P, 8);
  AttnArgs& aa = ap->aa;
  aa = AttnArgs{};
  aa.B = B; aa.P = P; aa.H = c.horizon; aa.n_q = c.n_q_heads; aa.n_kv = nkv; aa.d_h = dh;
  aa.group = c.n_q_heads / nkv;
  aa.n_qt = cdiv(aa.group * c.horizon, 128);
  aa.cs = attn_cluster(P);
  aa.kc = attn_kc(P, aa.cs);
  aa.kc_s = round_up(c.horizon, 16);
  aa.scale_log2 = (float)(1.4426950408889634 / sqrt((double)dh));
  aa.o = (bf16*)o; aa.o32 = o32; aa.xo = h->xo; aa.xml = h->xml; aa.status = h->d_status;
  aa.pmask = h->pmask; aa.pmw = h->pmw;
  const unsigned fl = c.flags;
  const bool stream_ok = dh == 64 || dh == 128 || dh == 256;
  // The clustered form holds at most 128 keys per rank (prefix keys over
  // cs - 1 ranks, the action keys on the last) and gives each rank d_h / cs
  // output columns in whole 8-column groups; a longer prefix or horizon, or
  // too narrow a head for the cluster, takes the streaming form.
  const bool split_ok = aa.kc <= 128 && aa.kc_s <= 128 && (dh / aa.cs) % 8 == 0;
  ap->stream = stream_ok && ((fl & VLA_FLAG_ATTN_STREAM) ||
                             (!(fl & VLA_FLAG_ATTN_SPLIT) && (!split_ok || B * nkv * aa.n_qt * 5 >= h->num_sms)));
  const uint32_t krows = ap->stream ? 128u : (uint32_t)aa.kc, ksrows = ap->stream ? 128u : (uint32_t)aa.kc_s;
  if (tc_encode_2d_bf16(&ap->tmQ, h->q, dh, (uint64_t)B * c.n_q_heads * c.horizon, 64, 128) ||
      tc_encode_3d_bf16(&ap->tmK, kc, dh, P, (uint64_t)L * B * nkv, (uint64_t)dh * 2, (uint64_t)P * dh * 2, 64,
                        krows) ||
      tc_encode_3d_bf16(&ap->tmVt, vc, P, dh, (uint64_t)L * B * nkv, (uint64_t)P8 * 2, (uint64_t)dh * P8 * 2, 64,
                        dh) ||
      tc_encode_3d_bf16(&ap->tmKs, h->ks, dh, c.horizon, (uint64_t)B * nkv, (uint64_t)dh * 2,
                        (uint64_t)c.horizon * dh * 2, 64, ksrows) ||
      tc_encode_3d_bf16(&ap->tmVs, h->vs, c.horizon, dh, (uint64_t)B * nkv, (uint64_t)h->Hp * 2,
                        (uint64_t)dh * h->Hp * 2, 64, dh))
    return VLA_ERR_CUDA;
  return VLA_OK;
}

vla_status enqueue_attention(const vla_expert* h, const AttnPlan& ap, int layer, unsigned long long* tl,
                             cudaStream_t st) {
  AttnArgs aa = ap.aa;
  aa.layer = layer;
  aa.no_suffix = is_cross(h->cfg, layer) ? 1 : 0;
  aa.tl = tl;
  if (ap.stream) {
    VLA_CK(launch_attn_stream(&ap.tmQ, &ap.tmK, &ap.tmVt, &ap.tmKs, &ap.tmVs, aa, st));
  } else {
    VLA_CK(launch_attn_tc(&ap.tmQ, &ap.tmK, &ap.tmVt, &ap.tmKs, &ap.tmVs, aa, st));
  }
  return VLA_OK;
}

// The bf16 solver on the fused tensor-core kernels: per layer one QKV GEMM
// (norm prologue, scatter epilogue), the tcgen05 attention and its combine,
// the O GEMM (residual epilogue), the up GEMM (norm prologue, GeLU
// epilogue) and the down GEMM (residual epilogue); every launch uses
// programmatic dependent launch so weight streaming overlaps the previous
// kernel.
vla_status enqueue_denoise_fused(vla_expert* h, const void* kc, const void* vc, int B, int P, const float* noise,
                                 float* actions, float* tap, cudaStream_t st) {
  const vla_expert_config& c = h->cfg;
  const ExpertDims d = make_dims(h, B, P);
  const StepBufs sb = make_bufs(h, P);
  const int T = B * c.horizon, D = c.width, F = h->F_eff, L = c.n_layers;
  // Factored modulated norm: W u = r W((1 + gamma) h) + W beta.  Every
  // residual epilogue (and the input projection) writes (1 + gamma) h in
  // bf16 for the next normed map, whose epilogue applies the row scale r and
  // adds W beta (a per-(step, layer) table): no separate norm pass and no
  // norm prologue on the critical path of the next map.
  const bool fn = factored_norm(h);
  const LinPlan pq = plan_linear(h, h->qkvdim, D, T, !fn);
  const LinPlan po = plan_linear(h, D, h->qdim, T, false);
  const LinPlan pu = plan_linear(h, F, D, T, !fn);
  const LinPlan pd = plan_linear(h, D, F, T, false);
  bf16* act = (bf16*)h->act;
  CUtensorMap tm_uq, tm_uu, tm_o, tm_g;  // activations as B operands (box: 64 x the plan's BN)
  if (tc_encode_2d_bf16(&tm_uq, act, D, T, 64, pq.BN) || tc_encode_2d_bf16(&tm_uu, act, D, T, 64, pu.BN) ||
      tc_encode_2d_bf16(&tm_o, act, h->qdim, T, 64, po.BN) || tc_encode_2d_bf16(&tm_g, h->gbuf, F, T, 64, pd.BN))
    return VLA_ERR_CUDA;
  AttnPlan ap;
  VLA_ST(plan_attention(h, B, P, kc, vc, act, nullptr, &ap));
  CUtensorMap tmH;
  if (tc_encode_2d_f32(&tmH, h->h, D, T, 64, pq.BN)) return VLA_ERR_CUDA;
  CUtensorMap tm_xq, tm_xu;
  if (fn && (tc_encode_2d_bf16(&tm_xq, h->xt, D, T, 64, pq.BN) || tc_encode_2d_bf16(&tm_xu, h->xt, D, T, 64, pu.BN)))
    return VLA_ERR_CUDA;
  const DevCtl ctl{h->d_status, h->d_abort};
  const float* modt = h->modtab;
  for (int k = 0; k < h->S; ++k) {
    const float* x_in = k == 0 ? noise : actions;
    const float dt = step_dt(h, k);
    VLA_CK(launch_embed_ss(d, sb, x_in, h->ss2, ctl, st, fn ? h->xt : nullptr, modt + (size_t)k * L * 4 * D));
    int n_ss = embed_ss_slots(d);  // slots of ss2 currently valid
    for (int l = 0; l < L; ++l) {
      const float* mod = modt + ((size_t)k * L + l) * 4 * D;  // gamma_a, beta_a, gamma_m, beta_m
#ifdef VLA_TIMELINE
      // trace step 1, layers 1..4: slot (layer - 1) * 5 + kernel, 4096 CTAs x 16 events each
      auto tls = [&](int kidx) -> unsigned long long* {
        return (h->tl && k == 1 && l >= 1 && l <= 4) ? h->tl + ((size_t)((l - 1) * 5 + kidx)) * 4096 * 16 : nullptr;
      };
#else
      auto tls = [&](int) -> unsigned long long* { return nullptr; };
#endif
      // QKV
      LinArgs a = lin_args(h, pq, h->qkvdim, T, l);
      a.tl = tls(0);
      a.epi = EPI_QKV; a.q = (bf16*)h->q; a.ks = (bf16*)h->ks; a.vst = (bf16*)h->vs;
      if (fn) {
        a.fn_c = h->cqkv + ((size_t)k * L + l) * h->qkvdim; a.fn_ss = h->ss2; a.fn_nss = n_ss;
        if (!pq.wide) a.bmode = 2;
      } else if (pq.bmode == 1) {
        a.h_in = h->h; a.ss_in = h->ss2; a.n_ss_in = n_ss; a.gamma = mod; a.beta = mod + D;
      } else {
        VLA_CK(launch_modnorm(d, h->h, h->ss2, n_ss, mod, mod + D, act, st));
      }
      VLA_CK(run_lin(&h->tm_wqkv, fn ? &tm_xq : &tm_uq, &tmH, a, pq, st));
      // attention
      VLA_ST(enqueue_attention(h, ap, l, tls(1), st));
      // O projection + residual
      a = lin_args(h, po, D, T, l);
      a.epi = EPI_RESID; a.h = h->h; a.ss_out = h->ss1; a.tl = tls(2);
      // split O feeding a split up map: one statistics slot per rank
      const int nss_o = (fn && !po.wide && !pu.wide) ? po.tiles_n * po.C : po.tiles_n;
      if (fn) {
        a.xt_out = h->xt; a.xt_gamma = mod + 2 * D;
        if (!po.wide) a.bmode = 2;
        a.ss_per_rank = nss_o != po.tiles_n;
      }
      VLA_CK(run_lin(&h->tm_wo, &tm_o, &tmH, a, po, st));
      // MLP up + GeLU
      a = lin_args(h, pu, F, T, l);
      a.epi = EPI_GELU; a.g = (bf16*)h->gbuf; a.ldg = F; a.tl = tls(3);
      if (fn) {
        a.fn_c = h->cup + ((size_t)k * L + l) * F; a.fn_ss = h->ss1; a.fn_nss = nss_o;
        if (!pu.wide) a.bmode = 2;
      } else if (pu.bmode == 1) {
        a.h_in = h->h; a.ss_in = h->ss1; a.n_ss_in = po.tiles_n; a.gamma = mod + 2 * D; a.beta = mod + 3 * D;
      } else {
        VLA_CK(launch_modnorm(d, h->h, h->ss1, po.tiles_n, mod + 2 * D, mod + 3 * D, act, st));
      }
      VLA_CK(run_lin(&h->tm_wup, fn ? &tm_xu : &tm_uu, &tmH, a, pu, st));
      // MLP down + residual
      a = lin_args(h, pd, D, T, l);
      a.epi = EPI_RESID; a.h = h->h; a.ss_out = h->ss2; a.tl = tls(4);
      // split down feeding the next layer's split QKV map: one slot per rank
      const int nss_d = (fn && !pd.wide && !pq.wide) ? pd.tiles_n * pd.C : pd.tiles_n;
      if (fn && l + 1 < L) {  // the next layer's gamma_a
        a.xt_out = h->xt; a.xt_gamma = mod + 4 * D;
        if (!pd.wide) a.bmode = 2;
        a.ss_per_rank = nss_d != pd.tiles_n;
      }
      VLA_CK(run_lin(&h->tm_wdown, &tm_g, &tmH, a, pd, st));
      n_ss = a.ss_per_rank ? nss_d : pd.tiles_n;
    }
    VLA_CK(launch_head_fused(d, sb, k, dt, x_in, actions, tap, st));
  }
  return VLA_OK;
}

// The W2A8 solver on the tensor cores: per layer the Eq. (4) row quantiser
// before each of the four ternary maps (norm + quantise for QKV and up,
// quantise for the attention and GeLU outputs), the packed-ternary linear
// kernel with the (acc * alpha) * beta scaling fused into its epilogue, and
// the tcgen05 attention writing fp32 o for the quantiser.
vla_status enqueue_denoise_w2a8_fused(vla_expert* h, const void* kc, const void* vc, int B, int P, const float* noise,
                                      float* actions, float* tap, cudaStream_t st) {
  const vla_expert_config& c = h->cfg;
  const ExpertDims d = make_dims(h, B, P);
  const StepBufs sb = make_bufs(h, P);
  const int T = B * c.horizon, D = c.width, F = h->F_eff, L = c.n_layers, Q = h->qdim;
  const LinPlan pq = plan_linear(h, h->qkvdim, D, T, false);
  const LinPlan po = plan_linear(h, D, Q, T, false);
  const LinPlan pu = plan_linear(h, F, D, T, false);
  const LinPlan pd = plan_linear(h, D, F, T, false);
  bf16* act = (bf16*)h->act;
  CUtensorMap tm_u, tm_o, tm_g, tmH;
  if (tc_encode_2d_bf16(&tm_u, act, D, T, 64, pq.BN) || tc_encode_2d_bf16(&tm_o, act, Q, T, 64, po.BN) ||
      tc_encode_2d_bf16(&tm_g, act, F, T, 64, pd.BN) || tc_encode_2d_f32(&tmH, h->h, D, T, 64, pq.BN))
    return VLA_ERR_CUDA;
  AttnPlan ap;
  VLA_ST(plan_attention(h, B, P, kc, vc, nullptr, h->f32buf, &ap));
  const DevCtl ctl{h->d_status, h->d_abort};
  size_t tsz[kTapTensors];
  tap_sizes(h, B, tsz);
  for (int k = 0; k < h->S; ++k) {
    const float* x_in = k == 0 ? noise : actions;
    const float dt = step_dt(h, k);
    const bool tapping = h->tap && k == h->tap_step;
    // tap: copy workspace tensor `src` into tensor `i` of layer `l`
    auto cp = [&](int l, int i, const void* src) -> cudaError_t {
      return tapping ? cudaMemcpyAsync(tap_at(h, B, l, i), src, tsz[i], cudaMemcpyDeviceToDevice, st) : cudaSuccess;
    };
    auto tp = [&](int l, int i) -> void* { return tapping ? (void*)tap_at(h, B, l, i) : nullptr; };
    VLA_CK(launch_embed_ss(d, sb, x_in, h->ss2, ctl, st));
    for (int l = 0; l < L; ++l) {
      const float* mod = h->modtab + ((size_t)k * L + l) * 4 * D;
#ifdef VLA_TIMELINE
      auto tls = [&](int kidx) -> unsigned long long* {
        return (h->tl && k == 1 && l >= 1 && l <= 4) ? h->tl + ((size_t)((l - 1) * 5 + kidx)) * 4096 * 16 : nullptr;
      };
#else
      auto tls = [&](int) -> unsigned long long* { return nullptr; };
#endif
      VLA_CK(cp(l, 0, h->h));
      VLA_CK(launch_quant_norm(d, h->h, mod, mod + D, act, h->alpha, (float*)tp(l, 1), st));
      VLA_CK(cp(l, 2, act));
      VLA_CK(cp(l, 3, h->alpha));
      LinArgs a = lin_args(h, pq, h->qkvdim, T, l);
      a.tl = tls(0);
      a.epi = EPI_QKV; a.q = (bf16*)h->q; a.ks = (bf16*)h->ks; a.vst = (bf16*)h->vs;
      a.accout = (int32_t*)tp(l, 4);
      VLA_CK(launch_linear(&h->tm_wqkv, &tm_u, &tmH, a, pq.tiles_n, pq.tiles_t, pq.C, st));
      VLA_CK(cp(l, 5, h->q));
      VLA_CK(cp(l, 6, h->ks));
      VLA_CK(cp(l, 7, h->vs));
      VLA_ST(enqueue_attention(h, ap, l, tls(1), st));
      VLA_CK(cp(l, 8, h->f32buf));
      VLA_CK(launch_quant_rows(T, Q, h->f32buf, act, h->alpha, st));
      VLA_CK(cp(l, 9, act));
      VLA_CK(cp(l, 10, h->alpha));
      a = lin_args(h, po, D, T, l);
      a.tl = tls(2);
      a.epi = EPI_RESID; a.h = h->h; a.ss_out = nullptr; a.beta_off = h->qkvdim;  // the quantiser reads h itself
      a.accout = (int32_t*)tp(l, 11);
      VLA_CK(launch_linear(&h->tm_wo, &tm_o, &tmH, a, po.tiles_n, po.tiles_t, po.C, st));
      VLA_CK(cp(l, 12, h->h));
      VLA_CK(launch_quant_norm(d, h->h, mod + 2 * D, mod + 3 * D, act, h->alpha, (float*)tp(l, 13), st));
      VLA_CK(cp(l, 14, act));
      VLA_CK(cp(l, 15, h->alpha));
      a = lin_args(h, pu, F, T, l);
      a.tl = tls(3);
      a.epi = EPI_GELU; a.g32 = h->f32buf; a.ldg = F; a.beta_off = h->qkvdim + D;
      a.accout = (int32_t*)tp(l, 16);
      VLA_CK(launch_linear(&h->tm_wup, &tm_u, &tmH, a, pu.tiles_n, pu.tiles_t, pu.C, st));
      VLA_CK(cp(l, 17, h->f32buf));
      VLA_CK(launch_quant_rows(T, F, h->f32buf, act, h->alpha, st));
      VLA_CK(cp(l, 18, act));
      VLA_CK(cp(l, 19, h->alpha));
      a = lin_args(h, pd, D, T, l);
      a.tl = tls(4);
      a.epi = EPI_RESID; a.h = h->h; a.ss_out = nullptr; a.beta_off = h->qkvdim + D + F;
      a.accout = (int32_t*)tp(l, 20);
      VLA_CK(launch_linear(&h->tm_wdown, &tm_g, &tmH, a, pd.tiles_n, pd.tiles_t, pd.C, st));
      VLA_CK(cp(l, 21, h->h));
    }
    VLA_CK(launch_head_fused(d, sb, k, dt, x_in, actions, tap, st));
  }
  return VLA_OK;
}

// ---------------------------------------------------------------------------
// Persistent whole-solve path (few tokens, bf16)
// ---------------------------------------------------------------------------
constexpr int kPersistMaxT = 64;

// Fills the per-call arguments; false when this (B, P) does not fit the
// persistent kernel's limits (B tiles per phase, TMEM columns, tokens).
bool persist_plan(const vla_expert* h, int B, int P, PersistArgs* pa) {
  const vla_expert_config& c = h->cfg;
  const int T = B * c.horizon, G = h->num_sms;
  if (!h->persist_ok || T > h->persist_T || h->F_eff != c.mlp_width || c.cross_every) return false;
  PersistArgs a{};
  a.L = c.n_layers; a.D = c.width; a.F = c.mlp_width; a.S = h->S; a.T = T; a.BN = round_up(T, 16);
  a.B = B; a.H = c.horizon; a.Hp = h->Hp; a.P = P; a.d_a = c.action_dim; a.d_h = c.head_dim;
  a.n_q = c.n_q_heads; a.n_kv = c.n_kv_heads;
  a.group = c.n_q_heads / c.n_kv_heads; a.qdim = h->qdim; a.kvdim = h->kvdim; a.qkvdim = h->qkvdim;
  a.nqt = cdiv(a.group * c.horizon, 128);
  a.npch = cdiv(P, 128);
  a.nch = a.npch + cdiv(c.horizon, 128);
  a.att_units = B * c.n_kv_heads * a.nqt * a.nch;
  if ((size_t)a.att_units > h->p_units || a.nch > 16) return false;
  // attention CTAs: one per unit, at most a quarter of the SMs
  a.n_att = a.att_units < G / 4 ? a.att_units : G / 4;
  const int GL = G - a.n_att;
  if (T > GL) return false;
  const int NK[4][2] = {{h->qkvdim, c.width}, {c.width, h->qdim}, {c.mlp_width, c.width}, {c.width, c.mlp_width}};
  int work = 0;
  for (int ph = 0; ph < 4; ++ph) {
    a.N[ph] = NK[ph][0];
    a.nkb[ph] = NK[ph][1] / 64;
    a.U[ph] = (NK[ph][0] / 128) * a.nkb[ph];
    for (int cta = 0; cta < GL; ++cta) {  // limits of every linear CTA's unit range
      const int u0 = (int)((long)a.U[ph] * cta / GL), u1 = (int)((long)a.U[ph] * (cta + 1) / GL);
      if (u1 <= u0) continue;
      const int len = u1 - u0, ntiles = len < a.nkb[ph] ? len : a.nkb[ph];
      const int nseg = (u1 - 1) / a.nkb[ph] - u0 / a.nkb[ph] + 1;
      // TMEM columns of the segment accumulators; column constants in the head-row buffer
      if (nseg * a.BN > 256 || ntiles > 5 || 6 * 64 > c.width) return false;
      const int stg = ntiles * a.BN * 256 > nseg * a.BN * 512 ? ntiles * a.BN * 256 : nseg * a.BN * 512;
      const int need = ntiles * a.BN * 128 + stg;
      if (need > work) work = need;
    }
  }
  a.work_bytes = work;
  if (persist_ring_stages(c.width, work) < 4) return false;
  a.eps = c.rms_eps;
  a.dt_sign = c.schedule == VLA_SCHEDULE_REVERSE ? -1.f : 1.f;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
  a.win = h->win; a.wout = h->wout; a.modtab = h->modtab; a.modf = h->modf; a.cqkv = h->cqkv; a.cup = h->cup;
  a.h = h->h; a.accq = h->p_accq; a.accu = h->p_accu; a.rms = h->p_rms;
  a.q = (bf16*)h->q; a.ks = (bf16*)h->ks; a.vs = (bf16*)h->vs; a.o = (bf16*)h->act;
  a.opart = h->p_opart; a.oml = h->p_oml;
  a.bar = h->p_bar; a.stop = (int*)(h->p_bar + 1); a.status = h->d_status; a.abort = h->d_abort;
  a.pmask = h->pmask; a.pmw = h->pmw;
  *pa = a;
  return true;
}

vla_status enqueue_persist(vla_expert* h, const void* kc, const void* vc, const PersistArgs& base, const float* noise,
                           float* actions, float* tap, cudaStream_t st) {
  const vla_expert_config& c = h->cfg;
  PersistArgs a = base;
  a.noise = noise; a.actions = actions; a.vtap = tap;
#ifdef VLA_PERSIST_TRACE
  a.trace = h->tl;
#endif
  const int dh = c.head_dim, nkv = c.n_kv_heads, L = c.n_layers, P = a.P, B = a.B, P8 = round_up(P, 8);
  CUtensorMap m[15];
  m[0] = h->tm_wqkv; m[1] = h->tm_wo; m[2] = h->tm_wup; m[3] = h->tm_wdown;
  if (tc_encode_3d_bf16(&m[4], kc, dh, P, (uint64_t)L * B * nkv, (uint64_t)dh * 2, (uint64_t)P * dh * 2, 64, 128) ||
      tc_encode_3d_bf16(&m[5], vc, P, dh, (uint64_t)L * B * nkv, (uint64_t)P8 * 2, (uint64_t)dh * P8 * 2, 64, dh) ||
      tc_encode_3d_bf16(&m[6], h->ks, dh, c.horizon, (uint64_t)B * nkv, (uint64_t)dh * 2,
                        (uint64_t)c.horizon * dh * 2, 64, 128) ||
      tc_encode_3d_bf16(&m[7], h->vs, c.horizon, dh, (uint64_t)B * nkv, (uint64_t)h->Hp * 2,
                        (uint64_t)dh * h->Hp * 2, 64, dh) ||
      tc_encode_2d_bf16(&m[8], h->q, dh, (uint64_t)B * c.n_q_heads * c.horizon, 64, 128) ||
      tc_encode_2d_f32(&m[9], h->h, c.width, a.T, 64, a.BN) ||
      tc_encode_2d_f32(&m[10], h->p_accu, c.mlp_width, a.T, 64, a.BN) ||
      tc_encode_2d_bf16(&m[11], h->act, h->qdim, a.T, 64, a.BN) ||
      tc_encode_2d_f32(&m[12], h->p_accq, h->qkvdim, a.T, 128, a.T) ||
      tc_encode_2d_f32(&m[13], h->h, c.width, a.T, 128, a.T) ||
      tc_encode_2d_f32(&m[14], h->p_accu, c.mlp_width, a.T, 128, a.T))
    return VLA_ERR_CUDA;
  VLA_CK(launch_persist(m, a, h->num_sms, st));
  return VLA_OK;
}

vla_status validate_config(const vla_expert_config* c, int n_steps, bool w2a8) {
  if (!c || n_steps < 1) return VLA_ERR_INVALID_ARG;
  if (c->n_layers < 1 || c->width < 1 || c->mlp_width < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 ||
      c->head_dim < 1 || c->vlm_hidden < 1 || c->action_dim < 1 || c->horizon < 1 || c->time_dim < 2 ||
      c->max_batch < 1 || c->max_prefix < 1 || !(c->rms_eps > 0.f))
    return VLA_ERR_INVALID_ARG;
  if (c->dtype != VLA_DTYPE_F32 && c->dtype != VLA_DTYPE_BF16) return VLA_ERR_INVALID_ARG;
  if (c->schedule != VLA_SCHEDULE_FORWARD && c->schedule != VLA_SCHEDULE_REVERSE) return VLA_ERR_INVALID_ARG;
  if (c->cross_every < 0) return VLA_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads != 0 || c->time_dim % 2 != 0) return VLA_ERR_SHAPE;
  if (w2a8 && c->dtype != VLA_DTYPE_BF16) return VLA_ERR_INVALID_ARG;
  const int qdim = c->n_q_heads * c->head_dim;
  if (c->dtype == VLA_DTYPE_BF16 &&
      (c->width % 64 || c->mlp_width % 64 || qdim % 64 || c->vlm_hidden % 64))
    return VLA_ERR_UNSUPPORTED;
  if (c->action_dim > 1024 || c->width > 16384 || c->mlp_width > 32768 || qdim > 16384) return VLA_ERR_UNSUPPORTED;
  return VLA_OK;
}

vla_status create_common(const vla_expert_config* cfg, int n_steps, bool w2a8, cudaStream_t st, vla_expert** out) {
  vla_status s = validate_config(cfg, n_steps, w2a8);
  if (s != VLA_OK) return s;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return VLA_ERR_NO_DEVICE;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return VLA_ERR_NO_DEVICE;
  if (prop.major != 10 || prop.minor != 3) return VLA_ERR_NO_DEVICE;
  vla_expert* h = new (std::nothrow) vla_expert();
  if (!h) return VLA_ERR_OOM;
  h->cfg = *cfg;
  h->S = n_steps;
  h->w2a8 = w2a8;
  h->f32 = cfg->dtype == VLA_DTYPE_F32;
  h->es = h->f32 ? 4 : 2;
  h->use_tc = !h->f32 && !(cfg->flags & VLA_FLAG_SIMT_GEMM);
  h->num_sms = prop.multiProcessorCount;
  h->qdim = cfg->n_q_heads * cfg->head_dim;
  h->kvdim = cfg->n_kv_heads * cfg->head_dim;
  h->qkvdim = h->qdim + 2 * h->kvdim;
  h->Hp = round_up(cfg->horizon, 8);
  h->fused = fused_supported(*cfg, h->f32, w2a8, h->use_tc);
#if defined(VLA_TIMELINE) || defined(VLA_PERSIST_TRACE)
  VLA_CK(cudaMalloc((void**)&h->tl, (size_t)20 * 4096 * 16 * 8));
  VLA_CK(cudaMemset(h->tl, 0, (size_t)20 * 4096 * 16 * 8));
#endif
  h->F_eff = cfg->mlp_width;
  h->Kmax = cfg->width;
  if (cfg->mlp_width > h->Kmax) h->Kmax = cfg->mlp_width;
  if (h->qdim > h->Kmax) h->Kmax = h->qdim;
  *out = h;
  (void)st;
  VLA_CK(simt_kernels_init());
  VLA_CK(tc_kernels_init());
  VLA_CK(expert_kernels_init());
  VLA_CK(linear_kernels_init());
  VLA_CK(attn_kernels_init());
  VLA_CK(attn_stream_init());
  VLA_CK(linear_wide_init());
  VLA_CK(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
  return VLA_OK;
}

// Shared tail of create: time table, fp32 in/out maps, workspace, tensor maps.
vla_status finish_create(vla_expert* h, const void* wt1, const void* wt2, const void* wmod, const void* wmod_f,
                         const void* win, const void* wout, cudaStream_t st) {
  const vla_expert_config& c = h->cfg;
  const int L = c.n_layers, D = c.width, S = h->S, d_t = c.time_dim;
  const int wb = h->f32 ? 0 : 1;
  vla_status s;
  // fp32 copies of the tiny in/out projections
  if ((s = dalloc(&h->win, (size_t)D * c.action_dim * 4)) != VLA_OK) return s;
  if ((s = dalloc(&h->wout, (size_t)D * c.action_dim * 4)) != VLA_OK) return s;
  VLA_CK(launch_to_f32(win, wb, h->win, (size_t)D * c.action_dim, st));
  VLA_CK(launch_to_f32(wout, wb, h->wout, (size_t)D * c.action_dim, st));
  // time conditioning table for tau_k = k / S
  float *e = nullptr, *c1 = nullptr, *cc = nullptr;
  if ((s = dalloc(&e, (size_t)S * d_t * 4)) != VLA_OK) return s;
  if ((s = dalloc(&c1, (size_t)S * D * 4)) != VLA_OK) { cudaFree(e); return s; }
  if ((s = dalloc(&cc, (size_t)S * D * 4)) != VLA_OK) { cudaFree(e); cudaFree(c1); return s; }
  if ((s = dalloc(&h->modtab, (size_t)S * L * 4 * D * 4)) != VLA_OK) return s;
  if ((s = dalloc(&h->modf, (size_t)S * 2 * D * 4)) != VLA_OK) return s;
  cudaError_t err = launch_time_embed(e, S, d_t, c.schedule == VLA_SCHEDULE_REVERSE, st);
  if (err == cudaSuccess) err = launch_gemm_simt(0, e, d_t, wb, wt1, d_t, S, D, d_t, 1, c1, 0, D, nullptr, st);
  if (err == cudaSuccess) err = launch_silu(c1, (size_t)S * D, st);
  if (err == cudaSuccess) err = launch_gemm_simt(0, c1, D, wb, wt2, D, S, D, D, 1, cc, 0, D, nullptr, st);
  if (err == cudaSuccess) err = launch_silu(cc, (size_t)S * D, st);
  if (err == cudaSuccess)
    err = launch_gemm_simt(0, cc, D, wb, wmod, D, S, L * 4 * D, D, 1, h->modtab, 0, L * 4 * D, nullptr, st);
  if (err == cudaSuccess)
    err = launch_gemm_simt(0, cc, D, wb, wmod_f, D, S, 2 * D, D, 1, h->modf, 0, 2 * D, nullptr, st);
  if (err == cudaSuccess) err = cudaStreamSynchronize(st);
  cudaFree(e);
  cudaFree(c1);
  cudaFree(cc);
  VLA_CK(err);
  // workspace
  const int Tm = c.max_batch * c.horizon;
  const size_t ae = h->f32 ? 4 : 2;
  if ((s = dalloc(&h->h, (size_t)Tm * D * 4)) != VLA_OK) return s;
  if ((s = dalloc(&h->act, (size_t)Tm * h->Kmax * ae)) != VLA_OK) return s;
  if (h->w2a8) {
    if ((s = dalloc(&h->codes, (size_t)Tm * h->Kmax)) != VLA_OK) return s;
  }
  if ((s = dalloc(&h->alpha, (size_t)Tm * 4)) != VLA_OK) return s;
  size_t pe = 0;
  for (int B = 1; B <= c.max_batch; ++B) {
    const int T = B * c.horizon;
    for (int w = 0; w < 4; ++w) {
      int N, K;
      gemm_dims(h, w, &N, &K);
      const GemmPlan p = plan_gemm(h, N, K, T);
      const size_t need = (size_t)p.splits * T * N;
      if (need > pe) pe = need;
    }
  }
  h->part_elems = pe;
  if ((s = dalloc(&h->part, pe * 4)) != VLA_OK) return s;
  if ((s = dalloc(&h->q, (size_t)Tm * h->qdim * ae)) != VLA_OK) return s;
  if ((s = dalloc(&h->ks, (size_t)Tm * h->kvdim * ae)) != VLA_OK) return s;
  if ((s = dalloc(&h->vs, (size_t)c.max_batch * h->kvdim * h->Hp * ae)) != VLA_OK) return s;
  if (h->fused) {
    // sums of squares: at most one slot per (128-row tile of D, split rank)
    h->ss_elems = (size_t)(D / 128 * 16 + 8) * Tm;
    if ((s = dalloc(&h->ss1, h->ss_elems * 4)) != VLA_OK) return s;
    if ((s = dalloc(&h->ss2, h->ss_elems * 4)) != VLA_OK) return s;
    if ((s = dalloc(&h->gbuf, (size_t)Tm * c.mlp_width * 2)) != VLA_OK) return s;
    if (h->w2a8 && (s = dalloc(&h->f32buf, (size_t)Tm * (h->qdim > c.mlp_width ? h->qdim : c.mlp_width) * 4)) != VLA_OK)
      return s;
    // split-K exchange buffers: the largest plan over every batch size
    size_t xp = 0, xs = 0;
    for (int B = 1; B <= c.max_batch; ++B) {
      const int T = B * c.horizon;
      const int dims[4][3] = {{h->qkvdim, D, 1}, {D, h->qdim, 0}, {c.mlp_width, D, 1}, {D, c.mlp_width, 0}};
      for (auto& g3 : dims) {
        const LinPlan p = plan_linear(h, g3[0], g3[1], T, g3[2] != 0);
        const size_t tiles = (size_t)p.tiles_n * p.tiles_t * p.C;
        if (tiles * p.BN * 128 > xp) xp = tiles * p.BN * 128;
        if (tiles * p.BN > xs) xs = tiles * p.BN;
      }
    }
    h->xpart_elems = xp;
    h->xss_elems = xs;
    if ((s = dalloc(&h->xpart, xp * 4)) != VLA_OK) return s;
    if ((s = dalloc(&h->xss, xs * 4)) != VLA_OK) return s;
    const int cs = attn_cluster(c.max_prefix);
    const size_t qtiles = (size_t)c.max_batch * c.n_kv_heads * cdiv(c.n_q_heads / c.n_kv_heads * c.horizon, 128);
    if ((s = dalloc(&h->xo, qtiles * cs * 128 * c.head_dim * 2)) != VLA_OK) return s;
    if ((s = dalloc(&h->xml, qtiles * cs * 128 * sizeof(float2))) != VLA_OK) return s;
  }
  // attention key-chunk size: largest multiple of 16 (<= 128) whose staging fits
  ExpertDims dd = make_dims(h, 1, c.max_prefix);
  int chunk = 128;
  while (chunk > 16 && attention_smem_bytes(dd, chunk) > 200 * 1024) chunk -= 16;
  if (attention_smem_bytes(dd, chunk) > 220 * 1024) return VLA_ERR_UNSUPPORTED;
  h->attn_chunk = chunk;
  const int max_chunks = cdiv(c.max_prefix + c.horizon, chunk);
  if ((s = dalloc(&h->opart, (size_t)Tm * c.n_q_heads * max_chunks * c.head_dim * 4)) != VLA_OK) return s;
  if ((s = dalloc(&h->ml, (size_t)Tm * c.n_q_heads * max_chunks * 2 * 4)) != VLA_OK) return s;
  if ((s = dalloc(&h->d_status, 16)) != VLA_OK) return s;
  VLA_CK(cudaMemset(h->d_status, 0, 16));
  VLA_CK(cudaHostAlloc((void**)&h->h_abort, sizeof(int), cudaHostAllocMapped));
  *h->h_abort = 0;
  VLA_CK(cudaHostGetDevicePointer((void**)&h->d_abort, h->h_abort, 0));
  // TMA descriptors of the bf16 weights
  if (!h->f32) {
    const int N_kv = L * 2 * h->kvdim;
    if (tc_encode_2d_bf16(&h->tm_wkv, h->wkv_pre, c.vlm_hidden, N_kv, 64, 128)) return VLA_ERR_CUDA;
    if (h->w2a8) {
      if (tc_encode_2d_u8(&h->tm_wqkv, h->wqkv, D / 4, (uint64_t)L * h->qkvdim, 16, 128) ||
          tc_encode_2d_u8(&h->tm_wo, h->wo, h->qdim / 4, (uint64_t)L * D, 16, 128) ||
          tc_encode_2d_u8(&h->tm_wup, h->wup, D / 4, (uint64_t)L * c.mlp_width, 16, 128) ||
          tc_encode_2d_u8(&h->tm_wdown, h->wdown, c.mlp_width / 4, (uint64_t)L * D, 16, 128))
        return VLA_ERR_CUDA;
    } else {
      if (tc_encode_2d_bf16(&h->tm_wqkv, h->wqkv, D, (uint64_t)L * h->qkvdim, 64, 128)) return VLA_ERR_CUDA;
      if (tc_encode_2d_bf16(&h->tm_wo, h->wo, h->qdim, (uint64_t)L * D, 64, 128)) return VLA_ERR_CUDA;
      if (tc_encode_2d_bf16(&h->tm_wup, h->wup, D, (uint64_t)L * c.mlp_width, 64, 128)) return VLA_ERR_CUDA;
      if (tc_encode_2d_bf16(&h->tm_wdown, h->wdown, c.mlp_width, (uint64_t)L * D, 64, 128)) return VLA_ERR_CUDA;
    }
  }
  // W beta for every (step, layer): the beta half of the factored modulated
  // norm, used by the many-token linears and by the persistent solver
  auto wbeta_tables = [&]() -> vla_status {
    if (h->cqkv) return VLA_OK;
    const int F = c.mlp_width;
    vla_status s2;
    if ((s2 = dalloc(&h->cqkv, (size_t)S * L * h->qkvdim * 4)) != VLA_OK) return s2;
    if ((s2 = dalloc(&h->cup, (size_t)S * L * F * 4)) != VLA_OK) return s2;
    cudaError_t e2 = cudaSuccess;
    for (int l = 0; l < L && e2 == cudaSuccess; ++l) {
      e2 = launch_gemm_simt(0, h->modtab + ((size_t)l * 4 + 1) * D, L * 4 * D, 1,
                            (const char*)h->wqkv + (size_t)l * h->qkvdim * D * 2, D, S, h->qkvdim, D, 1,
                            h->cqkv + (size_t)l * h->qkvdim, 0, L * h->qkvdim, nullptr, st);
      if (e2 == cudaSuccess)
        e2 = launch_gemm_simt(0, h->modtab + ((size_t)l * 4 + 3) * D, L * 4 * D, 1,
                              (const char*)h->wup + (size_t)l * F * D * 2, D, S, F, D, 1, h->cup + (size_t)l * F, 0,
                              L * F, nullptr, st);
    }
    VLA_CK(e2);
    return VLA_OK;
  };
  if (h->fused && !h->w2a8 && !h->f32) {
    if ((s = wbeta_tables()) != VLA_OK) return s;
    if ((s = dalloc(&h->xt, (size_t)Tm * D * 2)) != VLA_OK) return s;
  }
  // persistent few-token solver: accumulators, attention partials
  const int dh = c.head_dim;
  if (h->fused && !h->w2a8 && !h->f32 && (c.flags & VLA_FLAG_PERSIST) && (dh == 64 || dh == 128 || dh == 256) &&
      D % 128 == 0 && c.mlp_width % 128 == 0 && h->qkvdim % 128 == 0 && h->qdim % 64 == 0 && c.action_dim <= 64 &&
      persist_att_fits(dh) && persist_smem_bytes(D) <= 227 * 1024) {
    int occ = 0;
    VLA_CK(persist_init());
    VLA_CK(persist_blocks_per_sm(D, &occ));
    const int Tp = occ >= 1 ? (Tm < kPersistMaxT ? Tm : kPersistMaxT) : 0;
    const int F = c.mlp_width;
    const int Bmax = Tp / c.horizon;
    if (Bmax >= 1) {
      h->persist_T = Tp;
      const int group = c.n_q_heads / c.n_kv_heads;
      h->p_units = (size_t)Bmax * c.n_kv_heads * cdiv(group * c.horizon, 128) *
                   (cdiv(c.max_prefix, 128) + cdiv(c.horizon, 128));
      if ((s = wbeta_tables()) != VLA_OK) return s;
      if ((s = dalloc(&h->p_accq, (size_t)Tp * h->qkvdim * 4)) != VLA_OK) return s;
      if ((s = dalloc(&h->p_accu, (size_t)Tp * F * 4)) != VLA_OK) return s;
      if ((s = dalloc(&h->p_rms, (size_t)2 * Tp * 4)) != VLA_OK) return s;
      // chunk partials [B*n_kv*nch][group*H] rows (at most 128 per unit)
      if ((s = dalloc(&h->p_opart, h->p_units * 128 * dh * 4)) != VLA_OK) return s;
      if ((s = dalloc(&h->p_oml, h->p_units * 128 * sizeof(float2))) != VLA_OK) return s;
      if ((s = dalloc(&h->p_bar, 64)) != VLA_OK) return s;
      VLA_CK(cudaMemset(h->p_bar, 0, 64));
      h->persist_ok = true;
    }
  }
  VLA_CK(cudaStreamSynchronize(st));
  return VLA_OK;
}

// dst[l] = [src_a[l]; src_b[l]; (src_c[l])]: stacks per-layer row blocks.
cudaError_t stack_rows(void* dst, size_t dst_pitch, const void* src, size_t rows_bytes, int L, size_t offset,
                       cudaStream_t st) {
  return cudaMemcpy2DAsync((char*)dst + offset, dst_pitch, src, rows_bytes, rows_bytes, L, cudaMemcpyDeviceToDevice,
                           st);
}

}  // namespace

extern "C" {

const char* vla_status_string(vla_status s) {
  switch (s) {
    case VLA_OK: return "ok";
    case VLA_ERR_INVALID_ARG: return "invalid argument";
    case VLA_ERR_SHAPE: return "inconsistent shape";
    case VLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case VLA_ERR_OOM: return "out of device memory";
    case VLA_ERR_CUDA: return "CUDA runtime error";
    case VLA_ERR_TIMEOUT: return "device wait timed out";
    case VLA_ERR_ABORTED: return "aborted";
    case VLA_ERR_NO_DEVICE: return "no sm_103 device";
  }
  return "unknown status";
}

const char* vla_version(void) { return "0.1.0"; }

const char* vla_last_error(void) { return g_last_error; }

#if defined(VLA_TIMELINE) || defined(VLA_PERSIST_TRACE)
// Copies the event trace (20 slots x 4096 CTAs x 16 events, ns) to the host.
int vla_debug_timeline(vla_expert* h, void* dst, size_t bytes) {
  if (!h || !h->tl || bytes > (size_t)20 * 4096 * 16 * 8) return 1;
  return cudaMemcpy(dst, h->tl, bytes, cudaMemcpyDeviceToHost) == cudaSuccess ? 0 : 5;
}
#endif

void vla_expert_destroy(vla_expert* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);
  if (h->wup_full) {  // a neuron selection is or was active: free the full weights
    h->wup = h->wup_full;
    h->wdown = h->wdown_full;
  }
  void* ptrs[] = {h->wkv_pre, h->wqkv, h->wo,   h->wup,   h->wdown, h->beta,  h->win,     h->wout,
                  h->modtab,  h->modf, h->h,    h->act,   h->codes, h->alpha, h->part,    h->q,
                  h->ks,      h->vs,   h->opart, h->ml,   h->d_status, h->req_z, h->req_kc, h->req_vc,
                  h->req_noise, h->req_act, h->ss1, h->ss2, h->aopart, h->aml, h->gbuf, h->tl, h->xpart, h->xss, h->xo, h->xml, h->f32buf,
                  h->cqkv, h->cup, h->p_accq, h->p_accu, h->p_rms, h->p_opart, h->p_oml, h->p_bar, h->noise_buf,
                  h->beta_rows, h->beta_pre_rows, h->zcodes, h->zalpha, h->wup_sel, h->wdown_sel, h->xt};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (h->h_abort) cudaFreeHost(h->h_abort);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  delete h;
}

vla_status vla_expert_create(const vla_expert_config* cfg, const vla_expert_weights* w, int n_steps, void* stream,
                             vla_expert** out) {
  if (!out || !w) return VLA_ERR_INVALID_ARG;
  *out = nullptr;
  const void* ptrs[] = {w->wk_pre, w->wv_pre, w->wq, w->wk, w->wv, w->wo, w->wup, w->wdown,
                        w->wmod,   w->win,    w->wout, w->wt1, w->wt2, w->wmod_f};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return VLA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  vla_expert* h = nullptr;
  vla_status s = create_common(cfg, n_steps, false, st, &h);
  if (s != VLA_OK) {
    vla_expert_destroy(h);
    return s;
  }
  const vla_expert_config& c = *cfg;
  const int L = c.n_layers, D = c.width, F = c.mlp_width;
  const size_t es = h->es;
  const size_t kvb = (size_t)h->kvdim * c.vlm_hidden * es;
  const size_t qb = (size_t)h->qdim * D * es, kb = (size_t)h->kvdim * D * es;
  cudaError_t e = cudaSuccess;
  if ((s = dalloc(&h->wkv_pre, 2 * kvb * L)) != VLA_OK || (s = dalloc(&h->wqkv, (qb + 2 * kb) * L)) != VLA_OK ||
      (s = dalloc(&h->wo, (size_t)D * h->qdim * es * L)) != VLA_OK ||
      (s = dalloc(&h->wup, (size_t)F * D * es * L)) != VLA_OK ||
      (s = dalloc(&h->wdown, (size_t)D * F * es * L)) != VLA_OK) {
    vla_expert_destroy(h);
    return s;
  }
  e = stack_rows(h->wkv_pre, 2 * kvb, w->wk_pre, kvb, L, 0, st);
  if (e == cudaSuccess) e = stack_rows(h->wkv_pre, 2 * kvb, w->wv_pre, kvb, L, kvb, st);
  if (e == cudaSuccess) e = stack_rows(h->wqkv, qb + 2 * kb, w->wq, qb, L, 0, st);
  if (e == cudaSuccess) e = stack_rows(h->wqkv, qb + 2 * kb, w->wk, kb, L, qb, st);
  if (e == cudaSuccess) e = stack_rows(h->wqkv, qb + 2 * kb, w->wv, kb, L, qb + kb, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->wo, w->wo, (size_t)D * h->qdim * es * L, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->wup, w->wup, (size_t)F * D * es * L, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->wdown, w->wdown, (size_t)D * F * es * L, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) {
    vla_expert_destroy(h);
    return cuda_status(e);
  }
  s = finish_create(h, w->wt1, w->wt2, w->wmod, w->wmod_f, w->win, w->wout, st);
  if (s != VLA_OK) {
    vla_expert_destroy(h);
    return s;
  }
  *out = h;
  return VLA_OK;
}

vla_status vla_expert_create_w2a8(const vla_expert_config* cfg, const vla_expert_weights_w2a8* w, int n_steps,
                                  void* stream, vla_expert** out) {
  if (!out || !w) return VLA_ERR_INVALID_ARG;
  *out = nullptr;
  const bool tpre = w->wk_pre_t || w->wv_pre_t;  // ternary prefix maps
  if (tpre && (!w->wk_pre_t || !w->wv_pre_t || !w->beta_wk_pre || !w->beta_wv_pre)) return VLA_ERR_INVALID_ARG;
  const void* ptrs[] = {w->wq, w->wk, w->wv, w->wo, w->wup, w->wdown, w->beta_wq,
                        w->beta_wk, w->beta_wv, w->beta_wo, w->beta_wup, w->beta_wdown, w->wmod, w->win,
                        w->wout, w->wt1, w->wt2, w->wmod_f};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return VLA_ERR_INVALID_ARG;
  if (tpre) {
    if (!aligned16(w->wk_pre_t) || !aligned16(w->wv_pre_t) || !aligned16(w->beta_wk_pre) || !aligned16(w->beta_wv_pre))
      return VLA_ERR_INVALID_ARG;
  } else if (!w->wk_pre || !w->wv_pre || !aligned16(w->wk_pre) || !aligned16(w->wv_pre)) {
    return VLA_ERR_INVALID_ARG;
  }
  if (cfg) {  // scale groups must divide every map's rows
    const int G = w->beta_group, qd = cfg->n_q_heads * cfg->head_dim, kd = cfg->n_kv_heads * cfg->head_dim;
    if (G < 0 || (G > 0 && (G % 4 || qd % G || kd % G || cfg->width % G || cfg->mlp_width % G))) return VLA_ERR_SHAPE;
  }
  cudaStream_t st = (cudaStream_t)stream;
  vla_expert* h = nullptr;
  vla_status s = create_common(cfg, n_steps, true, st, &h);
  if (s != VLA_OK) {
    vla_expert_destroy(h);
    return s;
  }
  const vla_expert_config& c = *cfg;
  const int L = c.n_layers, D = c.width, F = c.mlp_width, G = w->beta_group;
  const size_t kvb = tpre ? (size_t)h->kvdim * (c.vlm_hidden / 4) : (size_t)h->kvdim * c.vlm_hidden * 2;
  const size_t qb = (size_t)h->qdim * (D / 4), kb = (size_t)h->kvdim * (D / 4);
  const size_t ob = (size_t)D * (h->qdim / 4), ub = (size_t)F * (D / 4), db = (size_t)D * (F / 4);
  h->beta_stride = h->qkvdim + D + F + D;
  if ((s = dalloc(&h->wkv_pre, 2 * kvb * L)) != VLA_OK || (s = dalloc(&h->wqkv, (qb + 2 * kb) * L)) != VLA_OK ||
      (s = dalloc(&h->wo, ob * L)) != VLA_OK || (s = dalloc(&h->wup, ub * L)) != VLA_OK ||
      (s = dalloc(&h->wdown, db * L)) != VLA_OK || (s = dalloc(&h->beta, (size_t)L * 6 * 4)) != VLA_OK ||
      (s = dalloc(&h->beta_rows, (size_t)L * h->beta_stride * 4)) != VLA_OK ||
      (tpre && (s = dalloc(&h->beta_pre_rows, (size_t)L * 2 * h->kvdim * 4)) != VLA_OK)) {
    vla_expert_destroy(h);
    return s;
  }
  h->beta_group = G;
  h->tpre = tpre;
  cudaError_t e = stack_rows(h->wkv_pre, 2 * kvb, tpre ? (const void*)w->wk_pre_t : w->wk_pre, kvb, L, 0, st);
  if (e == cudaSuccess)
    e = stack_rows(h->wkv_pre, 2 * kvb, tpre ? (const void*)w->wv_pre_t : w->wv_pre, kvb, L, kvb, st);
  if (e == cudaSuccess) e = stack_rows(h->wqkv, qb + 2 * kb, w->wq, qb, L, 0, st);
  if (e == cudaSuccess) e = stack_rows(h->wqkv, qb + 2 * kb, w->wk, kb, L, qb, st);
  if (e == cudaSuccess) e = stack_rows(h->wqkv, qb + 2 * kb, w->wv, kb, L, qb + kb, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->wo, w->wo, ob * L, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->wup, w->wup, ub * L, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->wdown, w->wdown, db * L, cudaMemcpyDeviceToDevice, st);
  // scales: per output row, [L][q | k | v | o | up | down rows] (beta_{g(n)} of Eq. 4)
  const float* betas[6] = {w->beta_wq, w->beta_wk, w->beta_wv, w->beta_wo, w->beta_wup, w->beta_wdown};
  const int rows[6] = {h->qdim, h->kvdim, h->kvdim, D, F, D};
  int off = 0;
  for (int i = 0; i < 6 && e == cudaSuccess; ++i) {
    e = launch_expand_scales(h->beta_rows, betas[i], L, rows[i], G ? G : rows[i], h->beta_stride, off, st);
    off += rows[i];
  }
  if (G == 0)  // per-tensor table of the CUDA-core path
    for (int i = 0; i < 6 && e == cudaSuccess; ++i)
      e = cudaMemcpy2DAsync(h->beta + i, 6 * sizeof(float), betas[i], sizeof(float), sizeof(float), L,
                            cudaMemcpyDeviceToDevice, st);
  if (tpre && e == cudaSuccess) {  // prefix rows [L][K | V][kvdim]
    e = launch_expand_scales(h->beta_pre_rows, w->beta_wk_pre, L, h->kvdim, G ? G : h->kvdim, 2 * h->kvdim, 0, st);
    if (e == cudaSuccess)
      e = launch_expand_scales(h->beta_pre_rows, w->beta_wv_pre, L, h->kvdim, G ? G : h->kvdim, 2 * h->kvdim,
                               h->kvdim, st);
  }
  // reject packed bytes that hold the invalid code 3
  int* bad = nullptr;
  if (e == cudaSuccess) e = cudaMalloc((void**)&bad, sizeof(int));
  if (e == cudaSuccess) e = cudaMemsetAsync(bad, 0, sizeof(int), st);
  const void* packed[5] = {h->wqkv, h->wo, h->wup, h->wdown, h->wkv_pre};
  const size_t pbytes[5] = {(qb + 2 * kb) * L, ob * L, ub * L, db * L, 2 * kvb * L};
  for (int i = 0; i < (tpre ? 5 : 4) && e == cudaSuccess; ++i)
    e = launch_check_ternary_codes((const uint8_t*)packed[i], pbytes[i], bad, st);
  int hbad = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&hbad, bad, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (bad) cudaFree(bad);
  if (e != cudaSuccess) {
    vla_expert_destroy(h);
    return cuda_status(e);
  }
  if (hbad) {
    vla_expert_destroy(h);
    return VLA_ERR_INVALID_ARG;
  }
  if (tpre) {
    // the prefix rows' Eq. (4) codes (bf16 carriers) and scales for max_batch x max_prefix tokens
    const size_t rowsz = (size_t)c.max_batch * c.max_prefix;
    if ((s = dalloc(&h->zcodes, rowsz * c.vlm_hidden * 2)) != VLA_OK || (s = dalloc(&h->zalpha, rowsz * 4)) != VLA_OK) {
      vla_expert_destroy(h);
      return s;
    }
  }
  s = finish_create(h, w->wt1, w->wt2, w->wmod, w->wmod_f, w->win, w->wout, st);
  if (s != VLA_OK) {
    vla_expert_destroy(h);
    return s;
  }
  *out = h;
  return VLA_OK;
}

vla_status vla_prefix_cache_bytes(const vla_expert* h, int B, int P, size_t* bytes) {
  if (!h || !bytes || B < 1 || P < 1) return VLA_ERR_INVALID_ARG;
  // K_C [L][B][n_kv][P][d_h]; V_C^T [L][B][n_kv][d_h][P8] (the larger of the two)
  *bytes = (size_t)h->cfg.n_layers * B * h->cfg.n_kv_heads * round_up(P, 8) * h->cfg.head_dim * h->es;
  return VLA_OK;
}

vla_status vla_prefix_kv_build(vla_expert* h, const void* Z, int B, int P, void* Kc, void* Vc, void* stream) {
  if (!h || !Z || !Kc || !Vc || !aligned16(Z) || !aligned16(Kc) || !aligned16(Vc)) return VLA_ERR_INVALID_ARG;
  if (B < 1 || B > h->cfg.max_batch || P < 1 || P > h->cfg.max_prefix) return VLA_ERR_INVALID_ARG;
  const vla_expert_config& c = h->cfg;
  cudaStream_t st = (cudaStream_t)stream;
  const int BP = B * P, N = c.n_layers * 2 * h->kvdim, K = c.vlm_hidden;
  KvScatter kv{Kc, Vc, c.n_layers, B, c.n_kv_heads, P, c.head_dim, round_up(P, 8)};
  if (h->tpre) {
    // Ternary prefix maps (Eq. 4): quantise every prefix row of Z once, then
    // one packed-ternary product over all layers' K and V rows with the
    // cache scatter in its epilogue (no split: hundreds of row tiles).
    VLA_CK(launch_quant_rows_bf16(BP, K, (const bf16*)Z, (bf16*)h->zcodes, h->zalpha, st));
    LinArgs g{};
    g.N = N; g.T = BP; g.a_row0 = 0; g.KS = K; g.BN = BP >= 256 ? 256 : round_up(BP < 16 ? 16 : BP, 16);
    const int per_stage = 128 * 128 + g.BN * 128 + 128 * 16;
    g.stages = (200 * 1024) / per_stage;
    if (g.stages > 8) g.stages = 8;
    if (g.stages > K / 64) g.stages = K / 64;
    g.bmode = 0; g.amode = 1; g.w2a8 = 1; g.epi = EPI_KV;
    g.alpha = h->zalpha; g.wbeta = h->beta_pre_rows; g.beta_stride = 0; g.beta_off = 0; g.layer = 0;
    g.n_kv = c.n_kv_heads; g.d_h = c.head_dim; g.kvdim = h->kvdim;
    g.kc_out = (bf16*)Kc; g.vc_out = (bf16*)Vc; g.kv_B = B; g.kv_P = P; g.kv_P8 = round_up(P, 8);
    g.status = h->d_status; g.D = K;
    CUtensorMap tmA, tmB;
    if (tc_encode_2d_u8(&tmA, h->wkv_pre, K / 4, N, 16, 128) || tc_encode_2d_bf16(&tmB, h->zcodes, K, BP, 64, g.BN))
      return VLA_ERR_CUDA;
    VLA_CK(launch_linear(&tmA, &tmB, &tmB, g, cdiv(N, 128), cdiv(BP, g.BN), 1, st));
    return VLA_OK;
  }
  if (!h->use_tc) {
    VLA_CK(launch_gemm_simt(!h->f32, Z, K, !h->f32, h->wkv_pre, K, BP, N, K, 1, nullptr, 0, 0, &kv, st));
    return VLA_OK;
  }
  if (wide_applies(c.flags, h->num_sms, N, K, BP)) {
    // Many prefix tokens: the persistent kernel with the K / V^T scatter epilogue.
    const LinPlan p = plan_wide(h->num_sms, N, K, BP);
    CUtensorMap tmZw;
    if (tc_encode_2d_bf16(&tmZw, Z, K, BP, 64, p.BN)) return VLA_ERR_CUDA;
    LinArgs a{};
    a.N = N; a.T = BP; a.a_row0 = 0; a.KS = K; a.BN = p.BN; a.stages = p.stages; a.epi = EPI_KV;
    a.status = h->d_status;
    a.n_kv = c.n_kv_heads; a.d_h = c.head_dim; a.kvdim = h->kvdim;
    a.kc_out = (bf16*)Kc; a.vc_out = (bf16*)Vc; a.kv_B = B; a.kv_P = P; a.kv_P8 = round_up(P, 8);
    VLA_CK(launch_linear_wide(&h->tm_wkv, &tmZw, a, p.grid, st));
    return VLA_OK;
  }
  const int BN = BP >= 256 ? 256 : round_up(BP < 16 ? 16 : BP, 16);
  CUtensorMap tmZ;
  if (tc_encode_2d_bf16(&tmZ, Z, K, BP, 64, BN)) return VLA_ERR_CUDA;
  TcGemmArgs a{};
  a.N = N; a.T = BP; a.a_row0 = 0; a.num_kb = K / 64; a.kb_per_split = a.num_kb; a.BN = BN;
  const int stage = 128 * 128 + BN * 128;
  a.stages = (220 * 1024) / stage > 8 ? 8 : (220 * 1024) / stage;
  a.mode = 1; a.kv = kv; a.status = h->d_status;
  VLA_CK(launch_gemm_tc(&h->tm_wkv, &tmZ, a, cdiv(N, 128), cdiv(BP, BN), 1, st));
  return VLA_OK;
}

static vla_status denoise_impl(vla_expert* h, bool w2a8, const void* Kc, const void* Vc, int B, int P,
                               const float* noise, float* actions, float* tap, void* stream,
                               const uint32_t* pmask = nullptr) {
  if (!h || h->w2a8 != w2a8) return VLA_ERR_INVALID_ARG;
  if (!Kc || !Vc || !noise || !actions || !aligned16(Kc) || !aligned16(Vc) || !aligned16(noise) ||
      !aligned16(actions) || (tap && !aligned16(tap)) || (pmask && ((uintptr_t)pmask & 3u)))
    return VLA_ERR_INVALID_ARG;
  if (B < 1 || B > h->cfg.max_batch || P < 1 || P > h->cfg.max_prefix) return VLA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  h->pmask = pmask;
  h->pmw = (P + 31) / 32;
  // Few tokens (bf16) with VLA_FLAG_PERSIST: the whole solve is one persistent kernel launch.
  PersistArgs pa;
  if (!w2a8 && !h->tap && !(h->cfg.flags & (VLA_FLAG_SIMT_GEMM | VLA_FLAG_ATTN_SPLIT | VLA_FLAG_ATTN_STREAM |
                                            VLA_FLAG_LINEAR_SPLIT | VLA_FLAG_LINEAR_WIDE)) &&
      persist_plan(h, B, P, &pa))
    return enqueue_persist(h, Kc, Vc, pa, noise, actions, tap, st);
  auto enqueue = [&](cudaStream_t s2) {
    if (h->fused)
      return h->w2a8 ? enqueue_denoise_w2a8_fused(h, Kc, Vc, B, P, noise, actions, tap, s2)
                     : enqueue_denoise_fused(h, Kc, Vc, B, P, noise, actions, tap, s2);
    if (h->w2a8 && h->beta_group) return VLA_ERR_UNSUPPORTED;  // the CUDA-core W2A8 path has per-tensor scales
    return enqueue_denoise(h, Kc, Vc, B, P, noise, actions, tap, s2);
  };
  if ((h->cfg.flags & VLA_FLAG_NO_GRAPH) || h->tap) return enqueue(st);
  GraphEntry* hit = nullptr;
  for (auto& g : h->graphs)
    if (g.B == B && g.P == P && g.pmask == pmask && g.kc == Kc && g.vc == Vc && g.noise == noise &&
        g.actions == actions && g.tap == tap)
      hit = &g;
  if (!hit) {
    if ((int)h->graphs.size() >= kMaxGraphs) {
      size_t lru = 0;
      for (size_t i = 1; i < h->graphs.size(); ++i)
        if (h->graphs[i].last_use < h->graphs[lru].last_use) lru = i;
      cudaGraphExecDestroy(h->graphs[lru].exec);
      h->graphs.erase(h->graphs.begin() + lru);
    }
    cudaGraph_t graph = nullptr;
    VLA_CK(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
    vla_status s = enqueue(h->cap_stream);
    cudaError_t e = cudaStreamEndCapture(h->cap_stream, &graph);
    if (s != VLA_OK) {
      if (graph) cudaGraphDestroy(graph);
      return s;
    }
    VLA_CK(e);
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    VLA_CK(e);
    h->graphs.push_back(GraphEntry{B, P, pmask, Kc, Vc, noise, actions, tap, exec, 0});
    hit = &h->graphs.back();
  }
  hit->last_use = ++h->tick;
  VLA_CK(cudaGraphLaunch(hit->exec, st));
  return VLA_OK;
}

vla_status vla_action_denoise(vla_expert* h, const void* Kc, const void* Vc, int B, int P, const float* noise,
                              float* actions, float* tap, void* stream) {
  return denoise_impl(h, false, Kc, Vc, B, P, noise, actions, tap, stream);
}

vla_status vla_action_denoise_w2a8(vla_expert* h, const void* Kc, const void* Vc, int B, int P, const float* noise,
                                   float* actions, float* tap, void* stream) {
  return denoise_impl(h, true, Kc, Vc, B, P, noise, actions, tap, stream);
}

vla_status vla_expert_select_ffn(vla_expert* h, const int32_t* idx, int F_sel, void* stream) {
  if (!h) return VLA_ERR_INVALID_ARG;
  const vla_expert_config& c = h->cfg;
  const int L = c.n_layers, D = c.width, F = c.mlp_width;
  if (h->w2a8 || h->f32 || !h->fused) return VLA_ERR_UNSUPPORTED;
  if (F_sel < 0 || F_sel > F || F_sel % 128 || (F_sel > 0 && (!idx || ((uintptr_t)idx & 3u)))) return VLA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (!h->wup_full) {
    h->wup_full = h->wup;
    h->wdown_full = h->wdown;
  }
  for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);  // graphs hold the old weight maps
  h->graphs.clear();
  if (F_sel == 0 || F_sel == F) {
    if (F_sel == F) {
      // every neuron: still validate and apply the order given
    } else {
      h->F_eff = F;
      h->wup = h->wup_full;
      h->wdown = h->wdown_full;
      if (tc_encode_2d_bf16(&h->tm_wup, h->wup, D, (uint64_t)L * F, 64, 128) ||
          tc_encode_2d_bf16(&h->tm_wdown, h->wdown, F, (uint64_t)L * D, 64, 128))
        return VLA_ERR_CUDA;
      return VLA_OK;
    }
  }
  vla_status s;
  if (!h->wup_sel && ((s = dalloc(&h->wup_sel, (size_t)L * F * D * 2)) != VLA_OK ||
                      (s = dalloc(&h->wdown_sel, (size_t)L * D * F * 2)) != VLA_OK))
    return s;
  int* bad = nullptr;
  VLA_CK(cudaMallocAsync((void**)&bad, sizeof(int), st));
  cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(int), st);
  if (e == cudaSuccess) e = launch_check_ffn_idx(idx, L, F, F_sel, bad, st);
  int hbad = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&hbad, bad, sizeof(int), cudaMemcpyDeviceToHost, st);
  cudaFreeAsync(bad, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  VLA_CK(e);
  if (hbad) return VLA_ERR_INVALID_ARG;  // nothing changed
  VLA_CK(launch_gather_ffn((const bf16*)h->wup_full, (const bf16*)h->wdown_full, (bf16*)h->wup_sel,
                           (bf16*)h->wdown_sel, idx, L, F, D, F_sel, st));
  h->F_eff = F_sel;
  h->wup = h->wup_sel;
  h->wdown = h->wdown_sel;
  if (tc_encode_2d_bf16(&h->tm_wup, h->wup, D, (uint64_t)L * F_sel, 64, 128) ||
      tc_encode_2d_bf16(&h->tm_wdown, h->wdown, F_sel, (uint64_t)L * D, 64, 128))
    return VLA_ERR_CUDA;
  return VLA_OK;
}

vla_status vla_noise_fill(unsigned long long seed, size_t n, float* out, void* stream) {
  if (!out || n < 1) return VLA_ERR_INVALID_ARG;
  VLA_CK(launch_noise(seed, n, out, (cudaStream_t)stream));
  return VLA_OK;
}

vla_status vla_action_denoise_ex(vla_expert* h, const void* Kc, const void* Vc, int B, int P, const vla_request* req,
                                 float* actions, float* tap, void* stream) {
  if (!h || !req) return VLA_ERR_INVALID_ARG;
  if (B < 1 || B > h->cfg.max_batch) return VLA_ERR_INVALID_ARG;
  const float* noise = req->noise_dev;
  cudaStream_t st = (cudaStream_t)stream;
  if (!noise) {
    // X^0 drawn in the library from the seed, into a handle-owned buffer
    const size_t n = (size_t)B * h->cfg.horizon * h->cfg.action_dim;
    if (!h->noise_buf) {
      vla_status s = dalloc(&h->noise_buf, (size_t)h->cfg.max_batch * h->cfg.horizon * h->cfg.action_dim * 4);
      if (s != VLA_OK) return s;
    }
    VLA_CK(launch_noise(req->seed, n, h->noise_buf, st));
    if (req->noise_out_dev) {
      if (!aligned16(req->noise_out_dev)) return VLA_ERR_INVALID_ARG;
      VLA_CK(cudaMemcpyAsync(req->noise_out_dev, h->noise_buf, n * 4, cudaMemcpyDeviceToDevice, st));
    }
    noise = h->noise_buf;
  }
  return denoise_impl(h, h->w2a8, Kc, Vc, B, P, noise, actions, tap, stream, req->prefix_mask_dev);
}

vla_status vla_expert_launch_count(const vla_expert* h, int B, int P, int* kernels) {
  if (!h || !kernels || B < 1 || P < 1) return VLA_ERR_INVALID_ARG;
  PersistArgs pa;
  if (!(h->cfg.flags & (VLA_FLAG_SIMT_GEMM | VLA_FLAG_ATTN_SPLIT | VLA_FLAG_ATTN_STREAM | VLA_FLAG_LINEAR_SPLIT |
                        VLA_FLAG_LINEAR_WIDE)) &&
      persist_plan(h, B, P, &pa)) {
    *kernels = 1;  // the persistent solve kernel
    return VLA_OK;
  }
  // per solver step: embed+norm, then per layer 4 GEMMs, reduce_qkv,
  // attention partials, attention combine, 2 residual/norm reductions (the
  // last layer's second one is the velocity head) and the GeLU reduction.
  if (h->fused && h->w2a8) {
    // per step: embed, head; per layer: 4 quantisers, 4 GEMMs, attention
    *kernels = h->S * (2 + 9 * h->cfg.n_layers);
  } else if (h->fused) {
    const int T = B * h->cfg.horizon, D = h->cfg.width;
    const bool fn = factored_norm(h);
    const LinPlan pq = plan_linear(h, h->qkvdim, D, T, !fn), pu = plan_linear(h, h->F_eff, D, T, !fn);
    const int extra = fn ? 0 : (pq.bmode == 0) + (pu.bmode == 0);
    // per step: embed, head; per layer: 4 GEMMs and the attention, plus the
    // standalone norms when neither the in-GEMM prologue nor the factored
    // form applies
    *kernels = h->S * (2 + (5 + extra) * h->cfg.n_layers);
  } else {
    *kernels = h->S * (1 + 10 * h->cfg.n_layers);
  }
  return VLA_OK;
}

vla_status vla_expert_poll_status(vla_expert* h, void* stream) {
  if (!h) return VLA_ERR_INVALID_ARG;
  VLA_CK(cudaStreamSynchronize((cudaStream_t)stream));
  int v = 0;
  VLA_CK(cudaMemcpy(&v, h->d_status, sizeof(int), cudaMemcpyDeviceToHost));
  if (v) VLA_CK(cudaMemset(h->d_status, 0, sizeof(int)));
  return v == 0 ? VLA_OK : (vla_status)v;
}

vla_status vla_expert_set_abort(vla_expert* h, int abort) {
  if (!h || !h->h_abort) return VLA_ERR_INVALID_ARG;
  *(volatile int*)h->h_abort = abort ? 1 : 0;
  return VLA_OK;
}

vla_status vla_policy_step_host(vla_expert* h, const void* Z_host, int B, int P, const float* noise_host,
                                float* actions_host, void* stream) {
  if (!h || !Z_host || !noise_host || !actions_host) return VLA_ERR_INVALID_ARG;
  const vla_expert_config& c = h->cfg;
  if (B < 1 || B > c.max_batch || P < 1 || P > c.max_prefix) return VLA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  vla_status s;
  if (!h->req_z) {
    const size_t cache = (size_t)c.n_layers * c.max_batch * c.n_kv_heads * round_up(c.max_prefix, 8) * c.head_dim * h->es;
    if ((s = dalloc(&h->req_z, (size_t)c.max_batch * c.max_prefix * c.vlm_hidden * h->es)) != VLA_OK ||
        (s = dalloc(&h->req_kc, cache)) != VLA_OK || (s = dalloc(&h->req_vc, cache)) != VLA_OK ||
        (s = dalloc(&h->req_noise, (size_t)c.max_batch * c.horizon * c.action_dim * 4)) != VLA_OK ||
        (s = dalloc(&h->req_act, (size_t)c.max_batch * c.horizon * c.action_dim * 4)) != VLA_OK)
      return s;
  }
  const size_t zb = (size_t)B * P * c.vlm_hidden * h->es;
  const size_t xb = (size_t)B * c.horizon * c.action_dim * 4;
  VLA_CK(cudaMemcpyAsync(h->req_z, Z_host, zb, cudaMemcpyHostToDevice, st));
  VLA_CK(cudaMemcpyAsync(h->req_noise, noise_host, xb, cudaMemcpyHostToDevice, st));
  if ((s = vla_prefix_kv_build(h, h->req_z, B, P, h->req_kc, h->req_vc, stream)) != VLA_OK) return s;
  if ((s = denoise_impl(h, h->w2a8, h->req_kc, h->req_vc, B, P, h->req_noise, h->req_act, nullptr, stream)) != VLA_OK)
    return s;
  VLA_CK(cudaMemcpyAsync(actions_host, h->req_act, xb, cudaMemcpyDeviceToHost, st));
  return vla_expert_poll_status(h, stream);
}

vla_status vla_w2a8_quantize_rows(const float* x, int M, int K, int8_t* a, float* alpha, void* stream) {
  if (!x || !a || !alpha || M < 1 || K < 1 || K > 53248) return VLA_ERR_INVALID_ARG;
  VLA_CK(expert_kernels_init());
  VLA_CK(launch_quant_rows_i8(M, K, x, a, alpha, (cudaStream_t)stream));
  return VLA_OK;
}

vla_status vla_debug_gelu_forms(const float* x, int n, float* exact, float* fast, void* stream) {
  if (!x || !exact || !fast || n < 1) return VLA_ERR_INVALID_ARG;
  VLA_CK(launch_gelu_forms(x, n, exact, fast, (cudaStream_t)stream));
  return VLA_OK;
}

vla_status vla_expert_set_wait_limit(vla_expert* h, unsigned long long limit_ns) {
  if (!h || !h->d_status) return VLA_ERR_INVALID_ARG;
  VLA_CK(cudaMemcpy(h->d_status + 2, &limit_ns, sizeof(limit_ns), cudaMemcpyHostToDevice));
  return VLA_OK;
}

vla_status vla_expert_check_wait_timeout(vla_expert* h, void* stream) {
  if (!h || !h->d_status) return VLA_ERR_INVALID_ARG;
  VLA_CK(launch_expire_wait(h->d_status, (cudaStream_t)stream));
  return VLA_OK;
}

vla_status vla_expert_w2a8_tap_bytes(const vla_expert* h, int B, size_t* bytes) {
  if (!h || !bytes || !h->w2a8 || B < 1 || B > h->cfg.max_batch) return VLA_ERR_INVALID_ARG;
  *bytes = tap_layer_bytes(h, B) * (size_t)h->cfg.n_layers;
  return VLA_OK;
}

vla_status vla_expert_set_w2a8_tap(vla_expert* h, int step, void* tap_dev, size_t bytes) {
  if (!h || !h->w2a8) return VLA_ERR_INVALID_ARG;
  if (!tap_dev) {
    h->tap = nullptr;
    h->tap_cap = 0;
    h->tap_step = -1;
    return VLA_OK;
  }
  if (!h->fused || !aligned16(tap_dev) || step < 0 || step >= h->S ||
      bytes < tap_layer_bytes(h, h->cfg.max_batch) * (size_t)h->cfg.n_layers)
    return VLA_ERR_INVALID_ARG;
  h->tap = tap_dev;
  h->tap_cap = bytes;
  h->tap_step = step;
  return VLA_OK;
}

vla_status vla_w2a8_ternary_gemm(const int8_t* a, const float* alpha, const uint8_t* q, float beta, int M, int N,
                                 int K, uint16_t* y, int32_t* acc, void* stream) {
  if (!a || !alpha || !q || !y || M < 1 || N < 1 || K < 64 || K % 64 || K > 65536 || N % 4) return VLA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  VLA_CK(cudaGetDevice(&dev));
  VLA_CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  VLA_CK(simt_kernels_init());
  VLA_CK(linear_kernels_init());
  // Tensor cores: int8 codes carried exactly in bf16, ternary codes decoded
  // to bf16 in shared memory, fp32 accumulation of integers below 2^24.
  const LinPlan p = plan_linear_sms(sms, N, K, M, false, true);
  const size_t tiles = (size_t)p.tiles_n * p.tiles_t * p.C;
  bf16* carriers = nullptr;
  float* xpart = nullptr;
  float* xss = nullptr;
  VLA_CK(cudaMallocAsync((void**)&carriers, (size_t)M * K * 2, st));
  cudaError_t e = cudaMallocAsync((void**)&xpart, tiles * p.BN * 128 * 4, st);
  if (e == cudaSuccess) e = cudaMallocAsync((void**)&xss, tiles * p.BN * 4, st);
  if (e == cudaSuccess) e = launch_i8_to_bf16(a, carriers, (size_t)M * K, st);
  CUtensorMap tmA, tmB;
  if (e == cudaSuccess && (tc_encode_2d_u8(&tmA, q, K / 4, N, 16, 128) ||
                           tc_encode_2d_bf16(&tmB, carriers, K, M, 64, p.BN)))
    e = cudaErrorInvalidValue;
  if (e == cudaSuccess) {
    LinArgs g{};
    g.N = N; g.T = M; g.a_row0 = 0; g.KS = p.KS; g.BN = p.BN; g.stages = p.stages; g.bmode = 0; g.amode = p.amode;
    g.epi = EPI_W2A8_OUT; g.w2a8 = 1; g.alpha = alpha; g.wbeta = nullptr; g.beta_val = beta;
    g.yout = y; g.accout = acc; g.xpart = xpart; g.xss = xss; g.D = K;
    e = launch_linear(&tmA, &tmB, &tmB, g, p.tiles_n, p.tiles_t, p.C, st);
  }
  if (carriers) cudaFreeAsync(carriers, st);
  if (xpart) cudaFreeAsync(xpart, st);
  if (xss) cudaFreeAsync(xss, st);
  VLA_CK(e);
  return VLA_OK;
}

}  // extern "C"
