// Per-token kernels of the action expert's solver step.
//
// One velocity evaluation v(X^k, tau_k, C) ("vla.cpp: A Unified Inference
// Runtime for Vision-Language-Action Models", §III-A Eq. (1)).
//
// Default (fused) path: the linear maps and the attention run in
// k_linear_tc.cu / k_linear_wide.cu / k_attn_*.cu with their epilogues fused;
// this file supplies the per-step input projection with its row statistics
// (k_embed_ss*), the velocity head with the Euler update (k_head_*), the
// standalone modulated RMSNorm (k_modnorm*), the Eq. (4) row quantisers of
// the W2A8 variant (k_quant_*), the time-conditioning table, the seeded
// noise, the selected-neuron gathers and the bounded-wait self-test.
//
// Unfused path (the fp32 configuration and the CUDA-core diagnostic), per
// layer:
//   GEMM qkv -> reduce_qkv -> attention (split over key chunks) -> combine
//   GEMM o   -> reduce_norm (residual, MLP norm)
//   GEMM up  -> reduce_gelu
//   GEMM down-> reduce_norm (residual, next layer's attention norm) | head
// The GEMMs (k_gemm_tc.cu / k_gemm_simt.cu) write fp32 split-K partials; the
// kernels here reduce them in a fixed order (deterministic), fuse the
// epilogue (residual add, time-modulated RMSNorm, exact GeLU, the W2A8 output
// scaling of Eq. (4)) and emit the next GEMM's input (bf16 / fp32, or the
// Eq. (4) int8 codes for the W2A8 variant).  Attention is Eq. (2) with the
// action tokens' own keys/values appended to the cached prefix ones.
#include <math.h>

#include "vla_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMultiTokens = 256;  // from this many tokens the embed / head CTAs take several tokens
constexpr int kEmbedThreads = 128;
// CTAs per token of the per-token input projection (each writes its own
// sum-of-squares slot; the slot buffer holds D / 128 + 1 of them).
int embed_split(const ExpertDims& d) {
  int s = d.D / 128;
  return s > 8 ? 8 : (s < 1 ? 1 : s);
}

// ---------------------------------------------------------------------------
// Time conditioning table (built once per handle; tau_k = k / S, or
// 1 - k / S for the reverse schedule)
// ---------------------------------------------------------------------------
__global__ void k_time_embed(float* e, int S, int d_t, int reverse) {
  const int k = blockIdx.x;
  const int half = d_t / 2;
  const double tau = reverse ? 1.0 - (double)k / (double)S : (double)k / (double)S;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double omega = pow(10000.0, -(double)i / (double)half);
    const double arg = 1000.0 * tau * omega;
    e[(size_t)k * d_t + i] = (float)sin(arg);
    e[(size_t)k * d_t + half + i] = (float)cos(arg);
  }
}

// X^0 ~ N(0, I) from a seed: element e is normal (e mod 4) of Philox4x64-10
// block e / 4 (key (seed, 0), counter (e / 4, 0, 0, 0); Salmon et al., SC
// 2011), each pair of 64-bit words giving two normals by the Box-Muller
// transform in fp64.  One thread per block of four.
__device__ __forceinline__ void philox4x64_10(uint64_t c[4], uint64_t k0, uint64_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t a0 = 0xD2E7470EE14C6C93ull, a1 = 0xCA5A826395121157ull;
    const uint64_t hi0 = __umul64hi(a0, c[0]), lo0 = a0 * c[0];
    const uint64_t hi1 = __umul64hi(a1, c[2]), lo1 = a1 * c[2];
    const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
    k0 += 0x9E3779B97F4A7C15ull;
    k1 += 0xBB67AE8584CAA73Bull;
  }
}
__global__ void k_noise(unsigned long long seed, size_t n, float* out) {
  const size_t blk = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (blk * 4 >= n) return;
  uint64_t c[4] = {(uint64_t)blk, 0ull, 0ull, 0ull};
  philox4x64_10(c, (uint64_t)seed, 0ull);
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const double u1 = (double)((c[2 * p] >> 11) + 1) * 0x1p-53;
    const double u2 = (double)(c[2 * p + 1] >> 11) * 0x1p-53;
    const double r = sqrt(-2.0 * log(u1));
    double sn, cs;
    sincos(2.0 * 3.14159265358979323846 * u2, &sn, &cs);
    const size_t e = blk * 4 + 2 * p;
    if (e < n) out[e] = (float)(r * cs);
    if (e + 1 < n) out[e + 1] = (float)(r * sn);
  }
}

__global__ void k_silu(float* x, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = x[i];
    x[i] = v / (1.f + expf(-v));
  }
}

// ---------------------------------------------------------------------------
// Shared epilogue: modulated RMSNorm of a row in shared memory, emitted as
// the next GEMM's input (TU) or, for W2A8, quantised per Eq. (4).
// ---------------------------------------------------------------------------
template <typename TU>
__device__ void emit_modnorm(const ExpertDims& d, const StepBufs& b, float* row, const float* gamma,
                             const float* beta, int t, float* red) {
  float ss = 0.f;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) ss += row[i] * row[i];
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / (float)d.D + d.eps);
  if (!d.w2a8) {
    TU* out = (TU*)b.act + (size_t)t * d.D;
    for (int i = threadIdx.x; i < d.D; i += blockDim.x) out[i] = from_f<TU>(row[i] * r * (1.f + gamma[i]) + beta[i]);
  } else {
    for (int i = threadIdx.x; i < d.D; i += blockDim.x) row[i] = row[i] * r * (1.f + gamma[i]) + beta[i];
    __syncthreads();
    const float alpha = quantize_row_block(row, d.D, b.codes + (size_t)t * d.D, nullptr, red);
    if (threadIdx.x == 0) b.alpha[t] = alpha;
  }
}

__device__ __forceinline__ const float* mod_ptr(const ExpertDims& d, const StepBufs& b, int step, int layer,
                                                int which) {
  // modtab [S][L][4][D]: which = 0 gamma_a, 1 beta_a, 2 gamma_m, 3 beta_m
  return b.modtab + (((size_t)step * d.L + layer) * 4 + which) * d.D;
}

// h = x W_in^T; u = modnorm(h) with layer 0's attention modulation.
template <typename TU>
__global__ void k_embed_norm(ExpertDims d, StepBufs b, int step, const float* x_in, DevCtl ctl) {
  extern __shared__ float sm[];
  float* row = sm;
  float* xs = sm + d.D;
  float* red = xs + d.d_a;
  const int t = blockIdx.x;
  if (t == 0 && threadIdx.x == 0 && ctl.abort && *ctl.abort) latch_error(ctl.status, VLA_DEV_ABORTED);
  for (int j = threadIdx.x; j < d.d_a; j += blockDim.x) xs[j] = x_in[(size_t)t * d.d_a + j];
  __syncthreads();
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) {
    const float* w = b.win + (size_t)i * d.d_a;
    float acc = 0.f;
    for (int j = 0; j < d.d_a; ++j) acc += xs[j] * w[j];
    row[i] = acc;
    b.h[(size_t)t * d.D + i] = acc;
  }
  __syncthreads();
  emit_modnorm<TU>(d, b, row, mod_ptr(d, b, step, 0, 0), mod_ptr(d, b, step, 0, 1), t, red);
}

// Sum the QKV split-K partials and scatter q / k_s / v_s into the
// per-(observation, head) layouts the attention kernel reads.
template <typename TQ>
__global__ void k_reduce_qkv(ExpertDims d, StepBufs b, int layer, int splits) {
  const int t = blockIdx.x;
  const int T = d.B * d.H;
  const int bb = t / d.H, i = t - bb * d.H;
  const int N = d.qkvdim;
  TQ* q = (TQ*)b.q;
  TQ* ks = (TQ*)b.ks;
  TQ* vs = (TQ*)b.vs;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    float s = 0.f;
    for (int z = 0; z < splits; ++z) s += b.part[((size_t)z * T + t) * N + n];
    const int slot = n < d.qdim ? 0 : (n < d.qdim + d.kvdim ? 1 : 2);
    if (d.w2a8) s = w2a8_scale(s, b.alpha[t], b.beta[layer * 6 + slot]);
    if (slot == 0) {
      const int j = n / d.d_h, e = n - j * d.d_h;
      q[(((size_t)bb * d.n_q + j) * d.H + i) * d.d_h + e] = from_f<TQ>(s);
    } else {
      const int nn = n - d.qdim - (slot == 2 ? d.kvdim : 0);
      const int g = nn / d.d_h, e = nn - g * d.d_h;
      if (slot == 1)
        ks[(((size_t)bb * d.n_kv + g) * d.H + i) * d.d_h + e] = from_f<TQ>(s);
      else
        vs[(((size_t)bb * d.n_kv + g) * d.d_h + e) * d.Hp + i] = from_f<TQ>(s);
    }
  }
}

// Eq. (2) over one chunk of the joint key list [prefix P ; suffix H] for one
// (observation, query head): unnormalised partial output, row max and sum.
template <typename TC, typename TQ>
__global__ void k_attn_part(ExpertDims d, StepBufs b, const TC* Kc, const TC* Vc) {
  extern __shared__ float sm[];
  const int H = d.H, dh = d.d_h, chunk = b.attn_chunk;
  float* qs = sm;                     // [H][dh], pre-scaled by 1/sqrt(d_h)
  float* Ks = qs + H * dh;            // [chunk][dh+1]
  float* Vs = Ks + chunk * (dh + 1);  // [chunk][dh]
  float* S = Vs + chunk * dh;         // [H][chunk]
  const int c = blockIdx.x, j = blockIdx.y, bb = blockIdx.z;
  const int g = j / (d.n_q / d.n_kv);
  const int nkeys = d.P + (b.no_suffix ? 0 : H);  // cross-attention layers: the cached keys only
  const int k0 = c * chunk;
  const int nk = min(chunk, nkeys - k0);
  const float scale = rsqrtf((float)dh);
  const TQ* qg = (const TQ*)b.q + ((size_t)bb * d.n_q + j) * H * dh;
  for (int idx = threadIdx.x; idx < H * dh; idx += blockDim.x) qs[idx] = to_f(qg[idx]) * scale;
  const TQ* ksg = (const TQ*)b.ks + ((size_t)bb * d.n_kv + g) * H * dh;
  const TQ* vsg = (const TQ*)b.vs + ((size_t)bb * d.n_kv + g) * dh * d.Hp;  // [d_h][Hp]
  const TC* Kg = Kc + ((size_t)bb * d.n_kv + g) * d.P * dh;
  const TC* Vg = Vc + ((size_t)bb * d.n_kv + g) * dh * d.P8;  // [d_h][P8]
  for (int idx = threadIdx.x; idx < nk * dh; idx += blockDim.x) {
    const int r = idx / dh, e = idx - r * dh;
    const int kk = k0 + r;
    float kv, vv;
    if (kk < d.P) {
      kv = to_f(Kg[(size_t)kk * dh + e]);
      vv = to_f(Vg[(size_t)e * d.P8 + kk]);
    } else {
      kv = to_f(ksg[(size_t)(kk - d.P) * dh + e]);
      vv = to_f(vsg[(size_t)e * d.Hp + (kk - d.P)]);
    }
    Ks[r * (dh + 1) + e] = kv;
    Vs[r * dh + e] = vv;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < H * nk; idx += blockDim.x) {
    const int t = idx / nk, r = idx - t * nk;
    const float* qr = qs + t * dh;
    const float* kr = Ks + r * (dh + 1);
    float s = 0.f;
    for (int e = 0; e < dh; ++e) s += qr[e] * kr[e];
    const int kk = k0 + r;  // a hidden prefix key: M = -inf in Eq. (2)
    if (b.pmask && kk < d.P && !((__ldg(b.pmask + (size_t)bb * b.pmw + (kk >> 5)) >> (kk & 31)) & 1u)) s = -INFINITY;
    S[t * chunk + r] = s;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float* ml = b.ml + (((size_t)bb * d.n_q + j) * b.n_chunks + c) * H * 2;
  for (int t = wid; t < H; t += nw) {
    float m = -INFINITY;
    for (int r = lane; r < nk; r += 32) m = fmaxf(m, S[t * chunk + r]);
    m = warp_max(m);
    float l = 0.f;
    for (int r = lane; r < nk; r += 32) {
      const float p = m == -INFINITY ? 0.f : expf(S[t * chunk + r] - m);  // a chunk of hidden keys
      S[t * chunk + r] = p;
      l += p;
    }
    l = warp_sum(l);
    if (lane == 0) {
      ml[t * 2 + 0] = m;
      ml[t * 2 + 1] = l;
    }
  }
  __syncthreads();
  float* op = b.opart + (((size_t)bb * d.n_q + j) * b.n_chunks + c) * H * dh;
  for (int idx = threadIdx.x; idx < H * dh; idx += blockDim.x) {
    const int t = idx / dh, e = idx - t * dh;
    const float* pr = S + t * chunk;
    float o = 0.f;
    for (int r = 0; r < nk; ++r) o += pr[r] * Vs[r * dh + e];
    op[idx] = o;
  }
}

// Merge the key-chunk partials of every head for one action token and emit
// the O-projection input row [n_q * d_h].
template <typename TU>
__global__ void k_attn_combine(ExpertDims d, StepBufs b) {
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + d.qdim;
  const int i = blockIdx.x, bb = blockIdx.y;
  const int t = bb * d.H + i;
  const int nc = b.n_chunks, H = d.H, dh = d.d_h;
  for (int idx = threadIdx.x; idx < d.qdim; idx += blockDim.x) {
    const int j = idx / dh, e = idx - j * dh;
    const size_t base = ((size_t)bb * d.n_q + j) * nc;
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, b.ml[((base + c) * H + i) * 2]);
    float num = 0.f, den = 0.f;
    for (int c = 0; c < nc; ++c) {
      const float* mlc = b.ml + ((base + c) * H + i) * 2;
      const float w = expf(mlc[0] - M);
      num += w * b.opart[((base + c) * H + i) * dh + e];
      den += w * mlc[1];
    }
    const float o = num / den;
    if (!d.w2a8)
      ((TU*)b.act)[(size_t)t * d.qdim + idx] = from_f<TU>(o);
    else
      row[idx] = o;
  }
  if (d.w2a8) {
    __syncthreads();
    const float alpha = quantize_row_block(row, d.qdim, b.codes + (size_t)t * d.qdim, nullptr, red);
    if (threadIdx.x == 0) b.alpha[t] = alpha;
  }
}

// h += sum_z part (W2A8: Eq. (4) output scaling first), then the modulated
// RMSNorm selected by (mod_layer, mod_half) emits the next GEMM input.
template <typename TU>
__global__ void k_reduce_norm(ExpertDims d, StepBufs b, int step, int beta_layer, int beta_slot, int mod_layer,
                              int mod_half, int splits) {
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + d.D;
  const int t = blockIdx.x;
  const int T = d.B * d.H;
  const float alpha = d.w2a8 ? b.alpha[t] : 0.f;
  const float beta = d.w2a8 ? b.beta[beta_layer * 6 + beta_slot] : 0.f;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) {
    float s = 0.f;
    for (int z = 0; z < splits; ++z) s += b.part[((size_t)z * T + t) * d.D + i];
    if (d.w2a8) s = w2a8_scale(s, alpha, beta);
    const float hv = b.h[(size_t)t * d.D + i] + s;
    b.h[(size_t)t * d.D + i] = hv;
    row[i] = hv;
  }
  __syncthreads();
  emit_modnorm<TU>(d, b, row, mod_ptr(d, b, step, mod_layer, 2 * mod_half),
                   mod_ptr(d, b, step, mod_layer, 2 * mod_half + 1), t, red);
}

// g = GeLU(sum_z part) (W2A8: GeLU of the Eq. (4) bf16 output, then quantise).
template <typename TU>
__global__ void k_reduce_gelu(ExpertDims d, StepBufs b, int layer, int splits) {
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + d.F;
  const int t = blockIdx.x;
  const int T = d.B * d.H;
  const float alpha = d.w2a8 ? b.alpha[t] : 0.f;
  const float beta = d.w2a8 ? b.beta[layer * 6 + 4] : 0.f;
  for (int n = threadIdx.x; n < d.F; n += blockDim.x) {
    float s = 0.f;
    for (int z = 0; z < splits; ++z) s += b.part[((size_t)z * T + t) * d.F + n];
    if (d.w2a8) s = w2a8_scale(s, alpha, beta);
    const float g = gelu_exact(s);
    if (!d.w2a8)
      ((TU*)b.act)[(size_t)t * d.F + n] = from_f<TU>(g);
    else
      row[n] = g;
  }
  if (d.w2a8) {
    __syncthreads();
    const float a = quantize_row_block(row, d.F, b.codes + (size_t)t * d.F, nullptr, red);
    if (threadIdx.x == 0) b.alpha[t] = a;
  }
}

// Last layer's residual, final modulated RMSNorm, velocity projection and
// the Euler update x <- x + dt v (Eq. (1)); optional velocity tap.
__global__ void k_head(ExpertDims d, StepBufs b, int step, int splits, float dt, const float* x_in, float* x_out,
                       float* tap) {
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + d.D;
  const int t = blockIdx.x;
  const int T = d.B * d.H;
  const float alpha = d.w2a8 ? b.alpha[t] : 0.f;
  const float beta = d.w2a8 ? b.beta[(d.L - 1) * 6 + 5] : 0.f;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) {
    float s = 0.f;
    for (int z = 0; z < splits; ++z) s += b.part[((size_t)z * T + t) * d.D + i];
    if (d.w2a8) s = w2a8_scale(s, alpha, beta);
    const float hv = b.h[(size_t)t * d.D + i] + s;
    row[i] = hv;
    ss += hv * hv;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / (float)d.D + d.eps);
  const float* gf = b.modf + (size_t)step * 2 * d.D;
  const float* bf = gf + d.D;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) row[i] = row[i] * r * (1.f + gf[i]) + bf[i];
  __syncthreads();
  // The d_a outputs are split over gridDim.y CTAs (each recomputes the
  // row's norm): at few tokens this spreads the W_out reads over more SMs.
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int per = (d.d_a + gridDim.y - 1) / gridDim.y;
  const int a0 = blockIdx.y * per, a1 = a0 + per < d.d_a ? a0 + per : d.d_a;
  for (int a = a0 + wid; a < a1; a += nw) {
    const float* w = b.wout + (size_t)a * d.D;
    float acc = 0.f;
    for (int i = lane; i < d.D; i += 32) acc += row[i] * w[i];
    acc = warp_sum(acc);
    if (lane == 0) {
      const size_t o = (size_t)t * d.d_a + a;
      x_out[o] = fmaf(dt, acc, x_in[o]);
      if (tap) tap[(size_t)step * T * d.d_a + o] = acc;
    }
  }
}

// h = x W_in^T and its row sum of squares (one slot) for the first layer's
// in-GEMM modulated RMSNorm; also latches the abort flag once per step.
// The D features of a token are split over gridDim.y CTAs (kEmbedSplit at few
// tokens, for parallelism); CTA y writes its partial sum of squares to slot
// y of ss_out [slots][T], which the next norm sums in fixed order.
// xt (nullable): also bf16((1 + xgam) h), the first layer's operand of the
// factored modulated norm (many-token linears).
__global__ void k_embed_ss(ExpertDims d, StepBufs b, const float* x_in, float* ss_out, DevCtl ctl, bf16* xt,
                           const float* xgam) {
  // The first kernel of a solver step waits before it lets the next kernel
  // start: the attention kernels load the prefix cache before their own
  // grid-dependency wait, so no early launch may reach back past the cache
  // build that precedes the solve.
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  extern __shared__ float sm[];
  float* xs = sm;
  float* red = sm + d.d_a;
  const int t = blockIdx.x;
  const int per = (d.D + gridDim.y - 1) / gridDim.y;
  const int i0 = blockIdx.y * per, i1 = i0 + per < d.D ? i0 + per : d.D;
  if (t == 0 && blockIdx.y == 0 && threadIdx.x == 0 && ctl.abort && *ctl.abort) latch_error(ctl.status, VLA_DEV_ABORTED);
  for (int j = threadIdx.x; j < d.d_a; j += blockDim.x) xs[j] = x_in[(size_t)t * d.d_a + j];
  __syncthreads();
  float ss = 0.f;
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const float* w = b.win + (size_t)i * d.d_a;
    float acc = 0.f;
    for (int j = 0; j < d.d_a; ++j) acc += xs[j] * w[j];
    b.h[(size_t)t * d.D + i] = acc;
    if (xt) xt[(size_t)t * d.D + i] = __float2bfloat16_rn((1.f + xgam[i]) * acc);
    ss += acc * acc;
  }
  ss = block_sum(ss, red);
  if (threadIdx.x == 0) ss_out[(size_t)blockIdx.y * (d.B * d.H) + t] = ss;
}

// Many-token form of k_embed_ss: a CTA takes kMT consecutive tokens, so each
// W_in row is read once per kMT tokens (the per-token form reads all of W_in
// for every token).  Same arithmetic per element.
constexpr int kMT = 16;
__global__ void k_embed_ss_multi(ExpertDims d, StepBufs b, const float* x_in, float* ss_out, DevCtl ctl, bf16* xt,
                                 const float* xgam) {
  // The first kernel of a solver step waits before it lets the next kernel
  // start: the attention kernels load the prefix cache before their own
  // grid-dependency wait, so no early launch may reach back past the cache
  // build that precedes the solve.
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  extern __shared__ float sm[];
  float* xs = sm;                // [kMT][d_a]
  float* red = sm + kMT * d.d_a; // [kMT][warps]
  const int T = d.B * d.H, t0 = blockIdx.x * kMT;
  const int nt = T - t0 < kMT ? T - t0 : kMT;
  const int nw = blockDim.x >> 5, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (blockIdx.x == 0 && threadIdx.x == 0 && ctl.abort && *ctl.abort) latch_error(ctl.status, VLA_DEV_ABORTED);
  for (int e = threadIdx.x; e < kMT * d.d_a; e += blockDim.x)
    xs[e] = e < nt * d.d_a ? x_in[(size_t)t0 * d.d_a + e] : 0.f;
  __syncthreads();
  float ss[kMT];
#pragma unroll
  for (int t = 0; t < kMT; ++t) ss[t] = 0.f;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) {
    const float* w = b.win + (size_t)i * d.d_a;
    float acc[kMT];
#pragma unroll
    for (int t = 0; t < kMT; ++t) acc[t] = 0.f;
    for (int j = 0; j < d.d_a; ++j) {
      const float wv = w[j];
#pragma unroll
      for (int t = 0; t < kMT; ++t) acc[t] += xs[t * d.d_a + j] * wv;
    }
    const float xg = xt ? 1.f + xgam[i] : 0.f;
#pragma unroll
    for (int t = 0; t < kMT; ++t)
      if (t < nt) {
        b.h[(size_t)(t0 + t) * d.D + i] = acc[t];
        if (xt) xt[(size_t)(t0 + t) * d.D + i] = __float2bfloat16_rn(xg * acc[t]);
        ss[t] += acc[t] * acc[t];
      }
  }
#pragma unroll
  for (int t = 0; t < kMT; ++t) {
    const float v = warp_sum(ss[t]);
    if (lane == 0) red[t * nw + wid] = v;
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    float v = 0.f;
    for (int w = 0; w < nw; ++w) v += red[threadIdx.x * nw + w];
    ss_out[t0 + threadIdx.x] = v;
  }
}

// u = h / rms(h) * (1 + gamma) + beta as bf16 [T][D], rms from n_ss slots.
__global__ void k_modnorm(int T, int D, float eps, const float* h, const float* ss, int n_ss, const float* gamma,
                          const float* beta, bf16* u) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int t = blockIdx.x;
  float s = 0.f;
  for (int k = 0; k < n_ss; ++k) s += ss[(size_t)k * T + t];
  const float r = rsqrtf(s / (float)D + eps);
  for (int i = threadIdx.x * 2; i < D; i += blockDim.x * 2) {
    const float2 hv = *(const float2*)(h + (size_t)t * D + i);
    const float v0 = hv.x * r * (1.f + gamma[i]) + beta[i];
    const float v1 = hv.y * r * (1.f + gamma[i + 1]) + beta[i + 1];
    *(uint32_t*)(u + (size_t)t * D + i) = pack_bf16x2(v0, v1);
  }
}

// Velocity head on the final residual stream + Euler update (Eq. (1)).
__global__ void k_head_fused(ExpertDims d, StepBufs b, int step, float dt, const float* x_in, float* x_out,
                             float* tap) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + d.D;
  const int t = blockIdx.x;
  const int T = d.B * d.H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) {
    const float hv = b.h[(size_t)t * d.D + i];
    row[i] = hv;
    ss += hv * hv;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / (float)d.D + d.eps);
  const float* gf = b.modf + (size_t)step * 2 * d.D;
  const float* bf = gf + d.D;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) row[i] = row[i] * r * (1.f + gf[i]) + bf[i];
  __syncthreads();
  // The d_a outputs are split over gridDim.y CTAs (each recomputes the
  // row's norm): at few tokens this spreads the W_out reads over more SMs.
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int per = (d.d_a + gridDim.y - 1) / gridDim.y;
  const int a0 = blockIdx.y * per, a1 = a0 + per < d.d_a ? a0 + per : d.d_a;
  for (int a = a0 + wid; a < a1; a += nw) {
    const float* w = b.wout + (size_t)a * d.D;
    float acc = 0.f;
    for (int i = lane; i < d.D; i += 32) acc += row[i] * w[i];
    acc = warp_sum(acc);
    if (lane == 0) {
      const size_t o = (size_t)t * d.d_a + a;
      x_out[o] = fmaf(dt, acc, x_in[o]);
      if (tap) tap[(size_t)step * T * d.d_a + o] = acc;
    }
  }
}

// Many-token form of k_head_fused: a CTA takes kHT tokens (one warp each for
// the norm), so each W_out row is read once per kHT tokens.
constexpr int kHT = 8;
__global__ void k_head_multi(ExpertDims d, StepBufs b, int step, float dt, const float* x_in, float* x_out,
                             float* tap) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  extern __shared__ float sm[];  // [kHT][D] modulated rows
  const int T = d.B * d.H, t0 = blockIdx.x * kHT;
  const int nt = T - t0 < kHT ? T - t0 : kHT;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float* gf = b.modf + (size_t)step * 2 * d.D;
  const float* bf = gf + d.D;
  for (int t = wid; t < kHT; t += nw) {
    float* row = sm + (size_t)t * d.D;
    if (t < nt) {
      const float* hr = b.h + (size_t)(t0 + t) * d.D;
      float ss = 0.f;
      for (int i = lane; i < d.D; i += 32) {
        const float hv = hr[i];
        row[i] = hv;
        ss += hv * hv;
      }
      ss = warp_sum(ss);
      const float r = rsqrtf(ss / (float)d.D + d.eps);
      for (int i = lane; i < d.D; i += 32) row[i] = row[i] * r * (1.f + gf[i]) + bf[i];
    } else {
      for (int i = lane; i < d.D; i += 32) row[i] = 0.f;
    }
  }
  __syncthreads();
  for (int a = wid; a < d.d_a; a += nw) {
    const float* w = b.wout + (size_t)a * d.D;
    float acc[kHT];
#pragma unroll
    for (int t = 0; t < kHT; ++t) acc[t] = 0.f;
    for (int i = lane; i < d.D; i += 32) {
      const float wv = w[i];
#pragma unroll
      for (int t = 0; t < kHT; ++t) acc[t] += sm[(size_t)t * d.D + i] * wv;
    }
#pragma unroll
    for (int t = 0; t < kHT; ++t) {
      const float v = warp_sum(acc[t]);
      if (lane == 0 && t < nt) {
        const size_t o = (size_t)(t0 + t) * d.d_a + a;
        x_out[o] = fmaf(dt, v, x_in[o]);
        if (tap) tap[(size_t)step * T * d.d_a + o] = v;
      }
    }
  }
}

// Eq. (4) on the modulated RMSNorm of h: one CTA per token computes the
// row's rms, u = h / rms * (1 + gamma) + beta, alpha = max(|u|, 1e-5) / 127
// and the codes (as exact bf16 carriers).
__global__ void k_quant_norm(int D, float eps, const float* h, const float* gamma, const float* beta, bf16* codes,
                             float* alpha, float* u_out) {
  // A few rows (batch 1): let the next kernel (a ternary linear) start its
  // weight prologue now, under this one; with many rows its early CTAs
  // would compete with this kernel's for the SMs.
  const bool early = gridDim.x <= 32;
  if (early && threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  if (!early && threadIdx.x == 0) griddep_launch_dependents();
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + D;
  const int t = blockIdx.x;
  float ss = 0.f;
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    const float v = h[(size_t)t * D + i];
    row[i] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / (float)D + eps);
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    row[i] = row[i] * r * (1.f + gamma[i]) + beta[i];
    if (u_out) u_out[(size_t)t * D + i] = row[i];
  }
  __syncthreads();
  const float al = quantize_row_block(row, D, nullptr, codes + (size_t)t * D, red);
  if (threadIdx.x == 0) alpha[t] = al;
}

// Eq. (4) on fp32 rows x [T][K]; codes as bf16 carriers (I8 false) or int8.
template <bool I8>
__global__ void k_quant_rows(int K, const float* x, void* codes, float* alpha) {
  // A few rows (batch 1): let the next kernel (a ternary linear) start its
  // weight prologue now, under this one; with many rows its early CTAs
  // would compete with this kernel's for the SMs.
  const bool early = gridDim.x <= 32;
  if (early && threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  if (!early && threadIdx.x == 0) griddep_launch_dependents();
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + K;
  const int t = blockIdx.x;
  for (int i = threadIdx.x; i < K; i += blockDim.x) row[i] = x[(size_t)t * K + i];
  __syncthreads();
  const float al = I8 ? quantize_row_block(row, K, (int8_t*)codes + (size_t)t * K, nullptr, red)
                      : quantize_row_block(row, K, nullptr, (bf16*)codes + (size_t)t * K, red);
  if (threadIdx.x == 0) alpha[t] = al;
}

// The same three row operations with the row held in registers: one CTA per
// row of K floats (K % 4 == 0), thread i owns the float4 columns i,
// i + blockDim.x, ... (RV of them), and every load of the row (and of gamma,
// beta) is issued before any of them is used, so a row costs one memory
// round trip.  RV = 1 (more threads per row) when there are few rows.
template <int RV>
__device__ __forceinline__ void load_row4(const float* p, int nc, float4 (&v)[RV]) {
  const float4* p4 = (const float4*)p;
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    v[k] = c < nc ? p4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// u = v * r * (1 + gamma) + beta, elementwise (the expression of the
// shared-memory kernels above).
__device__ __forceinline__ float4 modulate4(float4 v, float r, float4 g, float4 b) {
  return make_float4(v.x * r * (1.f + g.x) + b.x, v.y * r * (1.f + g.y) + b.y, v.z * r * (1.f + g.z) + b.z,
                     v.w * r * (1.f + g.w) + b.w);
}

// Eq. (4) codes of four values (exact integers carried in bf16), packed.
__device__ __forceinline__ uint2 codes4(float4 u, float al) {
  auto q = [&](float x) { return fminf(fmaxf(rintf(__fdiv_rn(x, al)), -128.f), 127.f); };
  return make_uint2(pack_bf16x2(q(u.x), q(u.y)), pack_bf16x2(q(u.z), q(u.w)));
}

// The same four codes as int8, packed little-endian into one word.
__device__ __forceinline__ uint32_t codes4_i8(float4 u, float al) {
  auto q = [&](float x) { return (uint32_t)((int)fminf(fmaxf(rintf(__fdiv_rn(x, al)), -128.f), 127.f) & 0xFF); };
  return q(u.x) | (q(u.y) << 8) | (q(u.z) << 16) | (q(u.w) << 24);
}

__device__ __forceinline__ float absmax4(float4 u) { return fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w))); }

template <int RV>
__global__ void k_modnorm_v(int T, int D, float eps, const float* h, const float* ss, int n_ss, const float* gamma,
                            const float* beta, bf16* u) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int t = blockIdx.x, nc = D >> 2;
  float4 v[RV], g[RV], b[RV];
  load_row4(h + (size_t)t * D, nc, v);
  load_row4(gamma, nc, g);
  load_row4(beta, nc, b);
  __shared__ float red[32];
  float s = 0.f;
  for (int k = threadIdx.x; k < n_ss; k += blockDim.x) s += ss[(size_t)k * T + t];
  s = block_sum(s, red);
  const float r = rsqrtf(s / (float)D + eps);
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    if (c < nc) {
      const float4 m = modulate4(v[k], r, g[k], b[k]);
      *(uint2*)(u + (size_t)t * D + 4 * c) = make_uint2(pack_bf16x2(m.x, m.y), pack_bf16x2(m.z, m.w));
    }
  }
}

// Eq. (4) on the modulated RMSNorm of h (the row's own sum of squares).
template <int RV>
__global__ void k_quant_norm_v(int D, float eps, const float* h, const float* gamma, const float* beta, bf16* codes,
                               float* alpha, float* u_out) {
  // A few rows (batch 1): let the next kernel (a ternary linear) start its
  // weight prologue now, under this one; with many rows its early CTAs
  // would compete with this kernel's for the SMs.
  const bool early = gridDim.x <= 32;
  if (early && threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  if (!early && threadIdx.x == 0) griddep_launch_dependents();
  __shared__ float red[32];
  const int t = blockIdx.x, nc = D >> 2;
  float4 v[RV], g[RV], b[RV];
  load_row4(h + (size_t)t * D, nc, v);
  load_row4(gamma, nc, g);
  load_row4(beta, nc, b);
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < RV; ++k) s += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
  s = block_sum(s, red);
  const float r = rsqrtf(s / (float)D + eps);
  float am = 0.f;
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    v[k] = modulate4(v[k], r, g[k], b[k]);
    const int c = threadIdx.x + k * blockDim.x;
    if (c < nc) {
      am = fmaxf(am, absmax4(v[k]));
      if (u_out) *(float4*)(u_out + (size_t)t * D + 4 * c) = v[k];
    }
  }
  am = block_max(am, red);
  const float al = __fdiv_rn(fmaxf(am, 1e-5f), 127.0f);
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    if (c < nc) *(uint2*)(codes + (size_t)t * D + 4 * c) = codes4(v[k], al);
  }
  if (threadIdx.x == 0) alpha[t] = al;
}

// Eq. (4) on fp32 rows x [T][K]; codes as bf16 carriers (I8 false) or int8.
template <int RV, bool I8>
__global__ void k_quant_rows_v(int K, const float* x, void* codes, float* alpha) {
  // A few rows (batch 1): let the next kernel (a ternary linear) start its
  // weight prologue now, under this one; with many rows its early CTAs
  // would compete with this kernel's for the SMs.
  const bool early = gridDim.x <= 32;
  if (early && threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  if (!early && threadIdx.x == 0) griddep_launch_dependents();
  __shared__ float red[32];
  const int t = blockIdx.x, nc = K >> 2;
  float4 v[RV];
  load_row4(x + (size_t)t * K, nc, v);
  float am = 0.f;
#pragma unroll
  for (int k = 0; k < RV; ++k) am = fmaxf(am, absmax4(v[k]));  // padding lanes hold zeros
  am = block_max(am, red);
  const float al = __fdiv_rn(fmaxf(am, 1e-5f), 127.0f);
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    if (c < nc) {
      if (I8)
        *(uint32_t*)((int8_t*)codes + (size_t)t * K + 4 * c) = codes4_i8(v[k], al);
      else
        *(uint2*)((bf16*)codes + (size_t)t * K + 4 * c) = codes4(v[k], al);
    }
  }
  if (threadIdx.x == 0) alpha[t] = al;
}

// Eq. (4) on bf16 rows (the prefix hidden states Z of the W2A8 prefix build):
// the same row quantiser on the exact fp32 values of the bf16 inputs.
__global__ void k_quant_rows_bf16(int K, const bf16* x, bf16* codes, float* alpha) {
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + K;
  const int t = blockIdx.x;
  for (int i = threadIdx.x; i < K; i += blockDim.x) row[i] = __bfloat162float(x[(size_t)t * K + i]);
  __syncthreads();
  const float al = quantize_row_block(row, K, nullptr, codes + (size_t)t * K, red);
  if (threadIdx.x == 0) alpha[t] = al;
}

// Per-output-row weight scales from per-group ones (beta_{g(n)} of Eq. (4)):
// dst[l * stride + off + n] = src[l * (N / G) + n / G].
__global__ void k_expand_scales(float* dst, const float* src, int L, int N, int G, int stride, int off) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x, l = blockIdx.y;
  if (n < N && l < L) dst[(size_t)l * stride + off + n] = src[(size_t)l * (N / G) + n / G];
}

// Selected FFN neurons (rMuscle's Action Cache): compact copies of the rows of
// W_up and the columns of W_down that idx [L][Fs] names (checked first by
// k_check_ffn_idx: every index in [0, F) and above its predecessor).
__global__ void k_check_ffn_idx(const int32_t* idx, int L, int F, int Fs, int* bad) {
  const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (i >= (size_t)L * Fs) return;
  const int j = (int)(i % Fs);
  const int n = idx[i];
  if (n < 0 || n >= F || (j > 0 && n <= idx[i - 1])) atomicExch(bad, 1);
}
__global__ void k_gather_up(const bf16* w, bf16* dst, const int32_t* idx, int L, int F, int D, int Fs) {
  const int j = blockIdx.x, l = blockIdx.y;
  const int n = idx[(size_t)l * Fs + j];
  if (n < 0 || n >= F) return;
  const uint4* src = (const uint4*)(w + ((size_t)l * F + n) * D);
  uint4* out = (uint4*)(dst + ((size_t)l * Fs + j) * D);
  for (int i = threadIdx.x; i < D / 8; i += blockDim.x) out[i] = src[i];
}
__global__ void k_gather_down(const bf16* w, bf16* dst, const int32_t* idx, int L, int F, int D, int Fs) {
  const int d = blockIdx.x, l = blockIdx.y;
  const bf16* src = w + ((size_t)l * D + d) * F;
  bf16* out = dst + ((size_t)l * D + d) * Fs;
  for (int j = threadIdx.x; j < Fs; j += blockDim.x) {
    const int n = idx[(size_t)l * Fs + j];
    out[j] = (n >= 0 && n < F) ? src[n] : __float2bfloat16_rn(0.f);
  }
}

// A bounded wait that cannot be satisfied: the mbarrier expects two arrivals
// and gets one.  The wait runs out after the handle's limit, latches
// VLA_DEV_TIMEOUT and the kernel returns (nothing is left in flight).
__global__ void k_expire_wait(int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 2);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(&bar);
    mbar_wait(&bar, 0, status);
  }
}

// Threads for a register-held row of K floats with RV float4 per thread,
// or 0 when the row does not fit.
int row_threads(int K, int RV) {
  if (K < 4 || K % 4 != 0) return 0;
  const int nc = K / 4;
  int th = (nc + RV - 1) / RV;
  th = (th + 31) / 32 * 32;
  return th <= 1024 ? th : 0;
}
// Few rows (a small batch): one float4 per thread where the row fits.
int row_vec(int rows, int K) { return rows < 256 && row_threads(K, 1) ? 1 : 2; }

__global__ void k_i8_to_bf16(const int8_t* a, bf16* out, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    out[i] = __float2bfloat16_rn((float)a[i]);
}

template <typename TS>
__global__ void k_to_f32(const TS* src, float* dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = to_f(src[i]);
}

}  // namespace

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
cudaError_t expert_kernels_init() {
  cudaError_t e = set_max_dyn_smem(k_attn_part<float, float>);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_attn_part<bf16, bf16>);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_reduce_gelu<float>);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_reduce_gelu<bf16>);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_quant_norm);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_quant_rows_bf16);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_quant_rows<false>);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_quant_rows<true>);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_attn_combine<float>);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_head_multi);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_head_fused);
  if (e != cudaSuccess) return e;
  e = set_max_dyn_smem(k_embed_ss_multi);
  if (e != cudaSuccess) return e;
  return set_max_dyn_smem(k_attn_combine<bf16>);
}

cudaError_t launch_to_f32(const void* src, int src_bf16, float* dst, size_t n, cudaStream_t st) {
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  if (src_bf16)
    k_to_f32<bf16><<<blocks, 256, 0, st>>>((const bf16*)src, dst, n);
  else
    k_to_f32<float><<<blocks, 256, 0, st>>>((const float*)src, dst, n);
  return cudaGetLastError();
}

static cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

int embed_ss_slots(const ExpertDims& d) { return d.B * d.H >= kMultiTokens && d.d_a <= 256 ? 1 : embed_split(d); }

cudaError_t launch_embed_ss(const ExpertDims& d, const StepBufs& b, const float* x_in, float* ss_out, DevCtl ctl,
                            cudaStream_t st, bf16* xt, const float* xgam) {
  ExpertDims dd = d;
  StepBufs bb = b;
  void* args[] = {&dd, &bb, (void*)&x_in, &ss_out, &ctl, &xt, (void*)&xgam};
  const int T = d.B * d.H;
  if (T >= kMultiTokens && d.d_a <= 256)
    return launch_pdl((const void*)k_embed_ss_multi, dim3((T + kMT - 1) / kMT), dim3(kThreads),
                      (size_t)(kMT * d.d_a + kMT * (kThreads / 32)) * sizeof(float), st, args);
  return launch_pdl((const void*)k_embed_ss, dim3(T, embed_split(d)), dim3(kEmbedThreads), (size_t)(d.d_a + 32) * sizeof(float),
                    st, args);
}

cudaError_t launch_modnorm(const ExpertDims& d, const float* h, const float* ss, int n_ss, const float* gamma,
                           const float* beta, bf16* u, cudaStream_t st) {
  int T = d.B * d.H, D = d.D;
  float eps = d.eps;
  void* args[] = {&T, &D, &eps, (void*)&h, (void*)&ss, &n_ss, (void*)&gamma, (void*)&beta, &u};
  const int rv = row_vec(T, D), th = row_threads(D, rv);
  if (th) return launch_pdl(rv == 1 ? (const void*)k_modnorm_v<1> : (const void*)k_modnorm_v<2>, dim3(T), dim3(th), 0, st, args);
  return launch_pdl((const void*)k_modnorm, dim3(T), dim3(kThreads), 0, st, args);
}

cudaError_t launch_quant_norm(const ExpertDims& d, const float* h, const float* gamma, const float* beta, bf16* codes,
                              float* alpha, float* u_out, cudaStream_t st) {
  int D = d.D;
  float eps = d.eps;
  void* args[] = {&D, &eps, (void*)&h, (void*)&gamma, (void*)&beta, &codes, &alpha, &u_out};
  const int rv = row_vec(d.B * d.H, D), th = row_threads(D, rv);
  if (th)
    return launch_pdl(rv == 1 ? (const void*)k_quant_norm_v<1> : (const void*)k_quant_norm_v<2>, dim3(d.B * d.H),
                      dim3(th), 0, st, args);
  return launch_pdl((const void*)k_quant_norm, dim3(d.B * d.H), dim3(512), (size_t)(D + 32) * sizeof(float), st, args);
}

static cudaError_t launch_quant_rows_any(int T, int K, const float* x, void* codes, bool i8, float* alpha,
                                         cudaStream_t st) {
  void* args[] = {&K, (void*)&x, &codes, &alpha};
  const int rv = row_vec(T, K), th = row_threads(K, rv);
  if (th) {
    const void* fn = rv == 1 ? (i8 ? (const void*)k_quant_rows_v<1, true> : (const void*)k_quant_rows_v<1, false>)
                             : (i8 ? (const void*)k_quant_rows_v<2, true> : (const void*)k_quant_rows_v<2, false>);
    return launch_pdl(fn, dim3(T), dim3(th), 0, st, args);
  }
  return launch_pdl(i8 ? (const void*)k_quant_rows<true> : (const void*)k_quant_rows<false>, dim3(T), dim3(512),
                    (size_t)(K + 32) * sizeof(float), st, args);
}

cudaError_t launch_quant_rows(int T, int K, const float* x, bf16* codes, float* alpha, cudaStream_t st) {
  return launch_quant_rows_any(T, K, x, codes, false, alpha, st);
}

cudaError_t launch_quant_rows_i8(int T, int K, const float* x, int8_t* codes, float* alpha, cudaStream_t st) {
  return launch_quant_rows_any(T, K, x, codes, true, alpha, st);
}

cudaError_t launch_quant_rows_bf16(int T, int K, const bf16* x, bf16* codes, float* alpha, cudaStream_t st) {
  const size_t smem = (size_t)(K + 32) * sizeof(float);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  k_quant_rows_bf16<<<T, 256, smem, st>>>(K, x, codes, alpha);
  return cudaGetLastError();
}

cudaError_t launch_expand_scales(float* dst, const float* src, int L, int N, int G, int stride, int off,
                                 cudaStream_t st) {
  k_expand_scales<<<dim3((N + 255) / 256, L), 256, 0, st>>>(dst, src, L, N, G, stride, off);
  return cudaGetLastError();
}

cudaError_t launch_check_ffn_idx(const int32_t* idx, int L, int F, int Fs, int* bad, cudaStream_t st) {
  const size_t n = (size_t)L * Fs;
  k_check_ffn_idx<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(idx, L, F, Fs, bad);
  return cudaGetLastError();
}

cudaError_t launch_gather_ffn(const bf16* wup, const bf16* wdown, bf16* up_sel, bf16* down_sel, const int32_t* idx,
                              int L, int F, int D, int Fs, cudaStream_t st) {
  k_gather_up<<<dim3(Fs, L), 128, 0, st>>>(wup, up_sel, idx, L, F, D, Fs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_gather_down<<<dim3(D, L), 256, 0, st>>>(wdown, down_sel, idx, L, F, D, Fs);
  return cudaGetLastError();
}

cudaError_t launch_expire_wait(int* status, cudaStream_t st) {
  k_expire_wait<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_i8_to_bf16(const int8_t* a, bf16* out, size_t n, cudaStream_t st) {
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  k_i8_to_bf16<<<blocks, 256, 0, st>>>(a, out, n);
  return cudaGetLastError();
}

cudaError_t launch_head_fused(const ExpertDims& d, const StepBufs& b, int step, float dt, const float* x_in,
                              float* x_out, float* tap, cudaStream_t st) {
  ExpertDims dd = d;
  StepBufs bb = b;
  void* args[] = {&dd, &bb, &step, &dt, (void*)&x_in, &x_out, &tap};
  const int T = d.B * d.H;
  if (T >= kMultiTokens && (size_t)kHT * d.D * sizeof(float) <= 200 * 1024)
    return launch_pdl((const void*)k_head_multi, dim3((T + kHT - 1) / kHT), dim3(kThreads),
                      (size_t)kHT * d.D * sizeof(float), st, args);
  const int split = d.d_a >= 32 ? 4 : 1;
  return launch_pdl((const void*)k_head_fused, dim3(T, split), dim3(kThreads), (size_t)(d.D + 32) * sizeof(float), st,
                    args);
}

cudaError_t launch_time_embed(float* e, int S, int d_t, int reverse, cudaStream_t st) {
  k_time_embed<<<S, 128, 0, st>>>(e, S, d_t, reverse);
  return cudaGetLastError();
}

cudaError_t launch_noise(unsigned long long seed, size_t n, float* out, cudaStream_t st) {
  const size_t blocks = (n + 3) / 4;
  k_noise<<<(unsigned)((blocks + 255) / 256), 256, 0, st>>>(seed, n, out);
  return cudaGetLastError();
}

cudaError_t launch_silu(float* x, size_t n, cudaStream_t st) {
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  k_silu<<<blocks, 256, 0, st>>>(x, n);
  return cudaGetLastError();
}

cudaError_t launch_embed_norm(const ExpertDims& d, const StepBufs& b, int step, const float* x_in, DevCtl ctl,
                              cudaStream_t st) {
  const size_t smem = (size_t)(d.D + d.d_a + 32) * sizeof(float);
  const int T = d.B * d.H;
  if (d.f32)
    k_embed_norm<float><<<T, kThreads, smem, st>>>(d, b, step, x_in, ctl);
  else
    k_embed_norm<bf16><<<T, kThreads, smem, st>>>(d, b, step, x_in, ctl);
  return cudaGetLastError();
}

cudaError_t launch_reduce_qkv(const ExpertDims& d, const StepBufs& b, int layer, int splits, cudaStream_t st) {
  const int T = d.B * d.H;
  if (d.f32)
    k_reduce_qkv<float><<<T, kThreads, 0, st>>>(d, b, layer, splits);
  else
    k_reduce_qkv<bf16><<<T, kThreads, 0, st>>>(d, b, layer, splits);
  return cudaGetLastError();
}

size_t attention_smem_bytes(const ExpertDims& d, int chunk) {
  return (size_t)(d.H * d.d_h + chunk * (2 * d.d_h + 1) + d.H * chunk) * sizeof(float);
}

cudaError_t launch_attention(const ExpertDims& d, const StepBufs& b, int layer, const void* kc, const void* vc,
                             cudaStream_t st) {
  const size_t layer_k = (size_t)d.B * d.n_kv * d.P * d.d_h;
  const size_t layer_v = (size_t)d.B * d.n_kv * d.d_h * d.P8;
  const size_t smem = attention_smem_bytes(d, b.attn_chunk);
  dim3 grid(b.n_chunks, d.n_q, d.B);
  if (d.f32)
    k_attn_part<float, float><<<grid, kThreads, smem, st>>>(d, b, (const float*)kc + layer * layer_k,
                                                          (const float*)vc + layer * layer_v);
  else
    k_attn_part<bf16, bf16><<<grid, kThreads, smem, st>>>(d, b, (const bf16*)kc + layer * layer_k,
                                                        (const bf16*)vc + layer * layer_v);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem2 = (size_t)(d.qdim + 32) * sizeof(float);
  dim3 grid2(d.H, d.B);
  if (d.f32)
    k_attn_combine<float><<<grid2, kThreads, smem2, st>>>(d, b);
  else
    k_attn_combine<bf16><<<grid2, kThreads, smem2, st>>>(d, b);
  return cudaGetLastError();
}

cudaError_t launch_reduce_norm(const ExpertDims& d, const StepBufs& b, int step, int beta_layer, int beta_slot,
                               int mod_layer, int mod_half, int splits, cudaStream_t st) {
  const int T = d.B * d.H;
  const size_t smem = (size_t)(d.D + 32) * sizeof(float);
  if (d.f32)
    k_reduce_norm<float><<<T, kThreads, smem, st>>>(d, b, step, beta_layer, beta_slot, mod_layer, mod_half, splits);
  else
    k_reduce_norm<bf16><<<T, kThreads, smem, st>>>(d, b, step, beta_layer, beta_slot, mod_layer, mod_half, splits);
  return cudaGetLastError();
}

cudaError_t launch_reduce_gelu(const ExpertDims& d, const StepBufs& b, int layer, int splits, cudaStream_t st) {
  const int T = d.B * d.H;
  const size_t smem = (size_t)(d.F + 32) * sizeof(float);
  if (d.f32)
    k_reduce_gelu<float><<<T, kThreads, smem, st>>>(d, b, layer, splits);
  else
    k_reduce_gelu<bf16><<<T, kThreads, smem, st>>>(d, b, layer, splits);
  return cudaGetLastError();
}

cudaError_t launch_head(const ExpertDims& d, const StepBufs& b, int step, int splits, float dt, const float* x_in,
                        float* x_out, float* tap, cudaStream_t st) {
  const int T = d.B * d.H;
  const size_t smem = (size_t)(d.D + 32) * sizeof(float);
  k_head<<<T, kThreads, smem, st>>>(d, b, step, splits, dt, x_in, x_out, tap);
  return cudaGetLastError();
}
