// Fused linear layer of the action expert for many tokens (batched
// requests), on tcgen05.  Same operation and epilogues as k_linear_tc.cu
// ("vla.cpp: A Unified Inference Runtime for Vision-Language-Action Models",
// §III-A Eq. (1): the velocity network of every Euler step; §III-B Eq. (2):
// queries and action keys/values for the joint attention):
//   y[t][n] = sum_k W[n][k] X[t][k]
// followed by EPI_QKV (scatter to q, k_s, v_s^T), EPI_RESID (h += y and the
// per-(128-row block, token) sums of squares of the new h), EPI_GELU
// (g = bf16(GeLU(y))) or EPI_KV (the prefix cache, §III-B Eq. (2): K_C and
// the transposed V_C of every layer from one GEMM over all layers' W_K, W_V).
//
// At batch 1 the layer is a weight stream and k_linear splits K over a
// cluster; with thousands of tokens it is a dense GEMM, and this kernel is a
// persistent, warp-specialised one:
//   warp 0      TMA producer: 128 x 64 weight and BN x 64 token tiles into a
//               four-stage ring (weights first, before the grid dependency
//               wait, for the CTA's first tile)
//   warp 1      MMA issuer: 128 x BN accumulator in one of two TMEM buffers
//   warps 2-9   epilogue: warp w reads TMEM lane quarter w % 4 (one output
//               row n per thread) and half (w - 2) / 4 of the token columns
// Each CTA takes tiles blockIdx.x, blockIdx.x + gridDim.x, ...; the epilogue
// of one tile runs while the MMAs of the next accumulate into the other TMEM
// buffer.  Tiles are ordered weight-tile fastest, so CTAs running at the same
// time share token tiles in L2.
#include "vla_common.cuh"

namespace {

constexpr uint32_t kWA = 128 * 128;  // one 128 x 64 bf16 weight stage
constexpr int kWS = 4;               // ring stages
constexpr int kEpiWarps = 8;
constexpr int kWideThreads = 64 + 32 * kEpiWarps;

struct WideSmem {
  uint32_t a, b, wss, stg, bars, slot, total;
};
constexpr int kStg = 32 * 34;  // bf16 staging elements per epilogue warp (32 x 32 chunk, rows padded to 34)
constexpr int kMaxSlots = 16;  // per-block sums of squares of a token (D <= 2048)

__host__ __device__ inline WideSmem wide_layout(int BN) {
  WideSmem s;
  s.a = 0;
  s.b = (uint32_t)kWS * kWA;
  s.wss = s.b + (uint32_t)kWS * (uint32_t)BN * 128u;  // [2 tile parities][2 halves][4 quarters][BN/2] fp32
  s.stg = s.wss + 16u * (uint32_t)(BN / 2) * 4u;      // [8 warps][kStg] bf16
  s.bars = s.stg + (uint32_t)kEpiWarps * kStg * 2u;
  s.slot = s.bars + (2 * kWS + 5) * 8;
  s.total = s.slot + 16;
  return s;
}

// After the call, lane l holds the sum over the warp's 32 lanes of v[l]
// (a transposing butterfly: 16 + 8 + 4 + 2 + 1 shuffles for 32 columns).
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) {
    const bool up = (lane & k) != 0;
#pragma unroll
    for (int j = 0; j < k; ++j) {
      const float send = up ? v[j] : v[j + k];
      const float keep = up ? v[j + k] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, k);
    }
  }
  return v[0];
}

// fp32 pairs: pack, unpack, multiply, fused multiply-add.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void up2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// GeLU x * Phi(x) with erf by Abramowitz & Stegun, Handbook of Mathematical
// Functions, formula 7.1.26 (|error of erf| <= 1.5e-7, far below the bf16
// rounding of the output): erf(z) ~ 1 - t (a1 + a2 t + ... + a5 t^4) e^(-z^2),
// t = 1 / (1 + p z), z >= 0, odd extension for negative arguments.
// Evaluated for two values at once: the FMA-pipe arithmetic on fp32 pairs
// (the reciprocal and the exponential stay per element), and the final
// product as h + h * erf with h = x / 2.
__device__ __forceinline__ void gelu_as7126_x2(float x0, float x1, float& g0, float& g1) {
  const uint64_t z = mul2(pk2(fabsf(x0), fabsf(x1)), pk2(0.70710678118654752f, 0.70710678118654752f));
  float d0, d1;
  up2(fma2(pk2(0.3275911f, 0.3275911f), z, pk2(1.f, 1.f)), d0, d1);
  const uint64_t t = pk2(__fdividef(1.f, d0), __fdividef(1.f, d1));
  uint64_t q = fma2(t, pk2(1.061405429f, 1.061405429f), pk2(-1.453152027f, -1.453152027f));
  q = fma2(t, q, pk2(1.421413741f, 1.421413741f));
  q = fma2(t, q, pk2(-0.284496736f, -0.284496736f));
  q = fma2(t, q, pk2(0.254829592f, 0.254829592f));
  q = mul2(t, q);
  float e0, e1;
  up2(mul2(mul2(z, z), pk2(-1.4426950408889634f, -1.4426950408889634f)), e0, e1);
  float tl0, tl1;
  up2(mul2(q, pk2(fast_exp2(e0), fast_exp2(e1))), tl0, tl1);  // 1 - erf(z)
  const uint64_t erfv = pk2(copysignf(1.f - tl0, x0), copysignf(1.f - tl1, x1));
  const uint64_t h = mul2(pk2(x0, x1), pk2(0.5f, 0.5f));
  up2(fma2(h, erfv, h), g0, g1);
}

// Both GeLU forms of the library side by side (for the unit check of the
// many-token epilogue's erf approximation against the erff form).
__global__ void k_gelu_forms(const float* x, int n, float* exact, float* fast) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x0 = x[i], x1 = i + 1 < n ? x[i + 1] : 0.f;
  float g0, g1;
  gelu_as7126_x2(x0, x1, g0, g1);
  exact[i] = gelu_exact(x0);
  fast[i] = g0;
  if (i + 1 < n) {
    exact[i + 1] = gelu_exact(x1);
    fast[i + 1] = g1;
  }
}

template <int EPI>
__global__ void __launch_bounds__(kWideThreads, 1)
    k_linear_wide(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const LinArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int BN = g.BN;
  const WideSmem Ls = wide_layout(BN);
  uint8_t* As = smem + Ls.a;
  uint8_t* Bs = smem + Ls.b;
  float* wss = (float*)(smem + Ls.wss);
  bf16* stg_all = (bf16*)(smem + Ls.stg);
  uint64_t* full = (uint64_t*)(smem + Ls.bars);
  uint64_t* empty = full + kWS;
  uint64_t* accf = empty + kWS;  // [2] accumulator ready (MMA commit)
  uint64_t* acce = accf + 2;     // [2] accumulator drained (epilogue threads)
  uint64_t* fin = acce + 2;      // every MMA of this CTA complete
  uint32_t* tmem_slot = (uint32_t*)(smem + Ls.slot);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_n = g.N / 128, tiles_t = (g.T + BN - 1) / BN, tiles = tiles_n * tiles_t;
  const int nkb = g.KS / 64;
  const uint32_t b_tile = (uint32_t)BN * 128u;

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < kWS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kEpiWarps * 32);
    }
    mbar_init(fin, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint32_t tx = kWA + b_tile;
      const int first = blockIdx.x;
      int pre = 0;
      if (first < tiles) {
        // Weights of the first tile: independent of the previous kernel.
        const int m0 = (first % tiles_n) * 128;
        pre = nkb < kWS ? nkb : kWS;
        for (int i = 0; i < pre; ++i) {
          mbar_arrive_expect_tx(&full[i], tx);
          tma_load_2d(As + (size_t)i * kWA, &tmA, &full[i], i * 64, g.a_row0 + m0);
        }
      }
      griddep_wait();
      int it = 0;
      bool okp = true;
      for (int tile = first; okp && tile < tiles; tile += gridDim.x) {
        const int m0 = (tile % tiles_n) * 128, t0 = (tile / tiles_n) * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kWS;
          if (it >= pre) {
            if (!mbar_wait(&empty[s], ((it / kWS) & 1) ^ 1, g.status)) {
              s_fail = 1;
              okp = false;
              break;
            }
            mbar_arrive_expect_tx(&full[s], tx);
            tma_load_2d(As + (size_t)s * kWA, &tmA, &full[s], kb * 64, g.a_row0 + m0);
          }
          tma_load_2d(Bs + (size_t)s * b_tile, &tmB, &full[s], kb * 64, t0);
        }
      }
      // Own copies land before the CTA can exit (normally all consumed).
      const int first_live = it > kWS ? it - kWS : 0;
      for (int i = first_live; i < it; ++i) mbar_drain(&full[i % kWS], (uint32_t)(i / kWS) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, BN);
      int it = 0, lt = 0;
      bool okm = true;
      for (int tile = blockIdx.x; okm && tile < tiles; tile += gridDim.x, ++lt) {
        const int buf = lt & 1;
        if (!mbar_wait(&acce[buf], ((lt >> 1) & 1) ^ 1, g.status)) {
          okm = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(buf * 256);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kWS;
          if (!mbar_wait(&full[s], (it / kWS) & 1, g.status)) {
            okm = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(As + (size_t)s * kWA);
          const uint32_t b_addr = smem_u32(Bs + (size_t)s * b_tile);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(dt, sdesc_k128(a_addr + k * 32), sdesc_k128(b_addr + k * 32), idesc, (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (okm) umma_commit(&accf[buf]);
      }
      if (!okm) s_fail = 1;
      umma_commit(fin);
      mbar_drain(fin, 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2-9) ----------------
    griddep_wait();  // reads and writes activations of earlier kernels
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);
    const int hbn = BN / 2;
    int slot = 0;  // q, k or v (EPI_QKV), from the tile's rows
    int lt = 0;
    // Factored norm (EPI_QKV / EPI_GELU with fn_c): epilogue thread fe owns
    // token fe of each tile's r table; the per-block sums of squares of the
    // next tile's token are loaded while the current tile is processed.
    const int fe = threadIdx.x - 64;
    float ssn[kMaxSlots];
    auto fetch_ss = [&](int tl) {
      const int tt = (tl / tiles_n) * BN + fe;
      const bool live = g.fn_c && tl < tiles && fe < BN && tt < g.T;
#pragma unroll
      for (int sl = 0; sl < kMaxSlots; ++sl)
        ssn[sl] = (live && sl < g.fn_nss) ? __ldcg(g.fn_ss + (size_t)sl * g.T + tt) : 0.f;
    };
    if (EPI == EPI_QKV || EPI == EPI_GELU) fetch_ss(blockIdx.x);
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++lt) {
      const int buf = lt & 1;
      const int m0 = (tile % tiles_n) * 128, t0 = (tile / tiles_n) * BN;
      const int n = m0 + row;
      const int tcols = (g.T - t0) < BN ? (g.T - t0) : BN;
      // Residual rows of this tile's columns (only this tile touches them):
      // the first chunk is fetched while the MMAs run, each next chunk
      // while the current one is processed.
      float hcur[32];
      auto load_h = [&](int cc, float (&hb)[32]) {
        const int nvv = tcols - cc;
        const float* hq = g.h + (size_t)(t0 + cc) * g.D + n;
#pragma unroll
        for (int j = 0; j < 32; ++j) hb[j] = j < nvv ? hq[(size_t)j * g.D] : 0.f;
      };
      // Factored norm: the next map's operand scale (EPI_RESID), or this
      // map's row scales r_t and W beta (EPI_QKV / EPI_GELU), fetched while
      // the MMAs run.
      float xg = 0.f, fc = 0.f;
      if (EPI == EPI_RESID && g.xt_out) xg = 1.f + g.xt_gamma[n];
      if ((EPI == EPI_QKV || EPI == EPI_GELU) && g.fn_c) {
        fc = g.fn_c[n];
        named_bar_sync(3, 32 * kEpiWarps);  // the previous tile's readers of the r table are done
        if (fe < BN) {  // token fe of this tile: its sums of squares were fetched one tile ahead
          float ssum = 0.f;
#pragma unroll
          for (int sl = 0; sl < kMaxSlots; ++sl) ssum += ssn[sl];
          wss[fe] = rsqrtf(ssum / (float)g.D + g.eps);
        }
        fetch_ss(tile + gridDim.x);
        named_bar_sync(3, 32 * kEpiWarps);
      }
      if (EPI == EPI_RESID) {
        // The whole tile's residual rows go to L2 while the MMAs run; the
        // first chunk is loaded into registers.
        const float* hq = g.h + (size_t)(t0 + half * hbn) * g.D + n;
        const int nh = tcols - half * hbn;
        for (int j = 0; j < hbn && j < nh; ++j) prefetch_l2(hq + (size_t)j * g.D);
        load_h(half * hbn, hcur);
      }
      const bool okw = __all_sync(0xffffffffu, mbar_wait(&accf[buf], (lt >> 1) & 1, g.status));
      tc_fence_after();
      if (EPI == EPI_QKV) slot = n < g.qdim ? 0 : (n < g.qdim + g.kvdim ? 1 : 2);
      // The warp's 32 output rows are consecutive features inside one head
      // of one of q, k, v (EPI_QKV) or of one layer's K or V (EPI_KV).
      const int nb = m0 + quarter * 32;  // the warp's first output row
      int kl = 0, kwhich = 0, khd = 0, ke0 = 0;
      if (EPI == EPI_KV) {
        kl = nb / (2 * g.kvdim);
        const int rem = nb - kl * 2 * g.kvdim;
        kwhich = rem / g.kvdim;
        const int r2 = rem - kwhich * g.kvdim;
        khd = r2 / g.d_h;
        ke0 = r2 - khd * g.d_h;
      }
      int qhd = 0, qd0 = 0;
      if (EPI == EPI_QKV) {
        const int rr = slot == 0 ? nb : (slot == 1 ? nb - g.qdim : nb - g.qdim - g.kvdim);
        qhd = rr / g.d_h;
        qd0 = rr - qhd * g.d_h;
      }
      // Token-major stores: lane l writes token (l >> 2) + 8 * pass of each
      // 32-token chunk; tdiv = H (EPI_QKV) or P (EPI_KV) splits a token
      // index into (observation, position) without a division per store.
      const int tdiv = EPI == EPI_KV ? g.kv_P : g.H;
      float* wq = wss + ((size_t)(buf * 2 + half) * 4 + quarter) * hbn;  // this warp's column sums
      const int hend = (half + 1) * hbn;  // BN is a multiple of 16: the last chunk of a half may be partial
      for (int c0 = half * hbn; c0 < hend; c0 += 32) {
        uint32_t r[32];
        if (okw) {
          tmem_ld16_nowait(tq + (uint32_t)(buf * 256 + c0), r);
          tmem_ld16_nowait(tq + (uint32_t)(buf * 256 + c0 + 16), r + 16);
          tmem_wait16(r);
          tmem_wait16(r + 16);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        // valid columns in this chunk (the 32 TMEM columns read stay inside the
        // tile's 256-column buffer: c0 + 32 <= hbn + 32 * ceil(hbn / 32) <= 256)
        const int lim = (tcols < hend ? tcols : hend) - c0;
        const int nv = okw ? (lim < 32 ? lim : 32) : 0;
        if (EPI == EPI_RESID) {
          const bool more = c0 + 32 < hend;
          float hnxt[32];
          if (more) load_h(c0 + 32, hnxt);
          float hv[32];
          float* hp = g.h + (size_t)(t0 + c0) * g.D + n;
          bf16* xp = g.xt_out + (size_t)(t0 + c0) * g.D + n;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            hv[j] = hcur[j] + __uint_as_float(r[j]);
            if (j < nv) {
              hp[(size_t)j * g.D] = hv[j];
              if (g.xt_out) xp[(size_t)j * g.D] = __float2bfloat16_rn(xg * hv[j]);
            }
            hv[j] = j < nv ? hv[j] * hv[j] : 0.f;
          }
          const float cs = warp_transpose_sum32(hv, lane);
          if (c0 + lane < hend) wq[c0 - half * hbn + lane] = cs;
          if (more) {
#pragma unroll
            for (int j = 0; j < 32; ++j) hcur[j] = hnxt[j];
          }
        } else {
          // GeLU and QKV: stage the warp's 32 x 32 bf16 chunk in shared
          // memory, then write whole rows.  The warp's 32 output rows are
          // consecutive features inside one head of one of q, k, v.
          bf16* stg = stg_all + (size_t)(warp - 2) * kStg;
          const bool vt = (EPI == EPI_QKV && slot == 2) || (EPI == EPI_KV && kwhich == 1);
          // the chunk's row scales r_t (factored norm) into registers before
          // any staging store (c0 is a multiple of 8: 16-byte aligned)
          float rc[32];
          if ((EPI == EPI_QKV || EPI == EPI_GELU) && g.fn_c) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 v4 = *(const float4*)(wss + c0 + 4 * q4);
              rc[4 * q4] = v4.x; rc[4 * q4 + 1] = v4.y; rc[4 * q4 + 2] = v4.z; rc[4 * q4 + 3] = v4.w;
            }
          }
          __syncwarp();
          if (!vt) {
            // token-major outputs (g, q, k): [col][row] so a token's 32 features are 64 contiguous bytes
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float y0 = __uint_as_float(r[j]), y1 = __uint_as_float(r[j + 1]);
              if ((EPI == EPI_QKV || EPI == EPI_GELU) && g.fn_c) {
                y0 = fmaf(rc[j], y0, fc);
                y1 = fmaf(rc[j + 1], y1, fc);
              }
              if (EPI == EPI_GELU) gelu_as7126_x2(y0, y1, y0, y1);
              stg[j * 32 + lane] = __float2bfloat16_rn(y0);
              stg[(j + 1) * 32 + lane] = __float2bfloat16_rn(y1);
            }
            __syncwarp();
            const int part = lane & 3;
            int tb = 0, ti = 0;  // (observation, position) of token t0 + c0 + (lane >> 2)
            if (EPI != EPI_GELU) {
              const int t = t0 + c0 + (lane >> 2);
              tb = t / tdiv;
              ti = t - tb * tdiv;
            }
#pragma unroll
            for (int pass = 0; pass < 4; ++pass) {  // 8 tokens per pass, 4 lanes x 16 bytes per token
              const int j = pass * 8 + (lane >> 2);
              if (j < nv) {
                const uint4 v = *(const uint4*)(stg + j * 32 + part * 8);
                bf16* dst;
                if (EPI == EPI_GELU) {
                  dst = g.g + (size_t)(t0 + c0 + j) * g.ldg + nb;
                } else if (EPI == EPI_KV) {
                  dst = g.kc_out + ((((size_t)kl * g.kv_B + tb) * g.n_kv + khd) * g.kv_P + ti) * g.d_h + ke0;
                } else {
                  dst = slot == 0 ? g.q + (((size_t)tb * g.n_q + qhd) * g.H + ti) * g.d_h + qd0
                                  : g.ks + (((size_t)tb * g.n_kv + qhd) * g.H + ti) * g.d_h + qd0;
                }
                *(uint4*)(dst + part * 8) = v;
              }
              if (EPI != EPI_GELU) {
                ti += 8;
                while (ti >= tdiv) {
                  ti -= tdiv;
                  ++tb;
                }
              }
            }
          } else {
            // v_s^T [B][n_kv][d_h][Hp] is token-contiguous per feature: stage
            // [row][col] (rows padded to 34 elements: conflict-free writes),
            // then one feature row of 32 tokens per warp store.
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              float y = __uint_as_float(r[j]);
              if (EPI == EPI_QKV && g.fn_c) y = fmaf(rc[j], y, fc);
              stg[lane * 34 + j] = __float2bfloat16_rn(y);
            }
            __syncwarp();
            const int t = t0 + c0 + lane;
            bf16* col;
            size_t pitch;
            if (EPI == EPI_KV) {
              const int b = t / g.kv_P, pp = t - b * g.kv_P;
              col = g.vc_out + ((((size_t)kl * g.kv_B + b) * g.n_kv + khd) * g.d_h + ke0) * g.kv_P8 + pp;
              pitch = (size_t)g.kv_P8;
            } else {
              const int b = t / g.H, i = t - b * g.H;
              col = g.vst + (((size_t)b * g.n_kv + qhd) * g.d_h + qd0) * g.Hp + i;
              pitch = (size_t)g.Hp;
            }
            if (lane < nv) {
#pragma unroll 4
              for (int rw = 0; rw < 32; ++rw) col[(size_t)rw * pitch] = stg[rw * 34 + lane];
            }
          }
        }
      }
      // TMEM buffer drained: the MMA warp may overwrite it.
      tc_fence_before();
      mbar_arrive(&acce[buf]);
      if (EPI == EPI_RESID) {
        // Sum the four quarters' column sums (fixed order) for this half.
        named_bar_sync(1 + half, 128);
        const int col = quarter * 32 + lane;  // column within the half
        if (okw && col < hbn && half * hbn + col < tcols) {
          const float* ws = wss + (size_t)(buf * 2 + half) * 4 * hbn;
          g.ss_out[(size_t)(tile % tiles_n) * g.T + t0 + half * hbn + col] =
              (ws[col] + ws[hbn + col]) + (ws[2 * hbn + col] + ws[3 * hbn + col]);
        }
      }
      if (!okw) s_fail = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t linear_wide_smem_bytes(int BN) { return 1024 + wide_layout(BN).total; }

cudaError_t launch_gelu_forms(const float* x, int n, float* exact, float* fast, cudaStream_t st) {
  const int pairs = (n + 1) / 2;
  k_gelu_forms<<<(pairs + 255) / 256, 256, 0, st>>>(x, n, exact, fast);
  return cudaGetLastError();
}

cudaError_t linear_wide_init() {
  cudaError_t e = set_max_dyn_smem(k_linear_wide<EPI_QKV>);
  if (e == cudaSuccess) e = set_max_dyn_smem(k_linear_wide<EPI_KV>);
  if (e == cudaSuccess) e = set_max_dyn_smem(k_linear_wide<EPI_RESID>);
  if (e == cudaSuccess) e = set_max_dyn_smem(k_linear_wide<EPI_GELU>);
  return e;
}

cudaError_t launch_linear_wide(const CUtensorMap* tmA, const CUtensorMap* tmB, const LinArgs& g, int grid,
                               cudaStream_t st) {
  if (g.BN < 64 || g.BN > 256 || g.BN % 16 || g.KS % 64 || g.KS < 64 || g.N % 128 || g.T < 1 || grid < 1 ||
      g.amode != 0 || g.w2a8 != 0 || (g.fn_c && (g.fn_nss < 1 || g.fn_nss > kMaxSlots || !g.fn_ss)) ||
      (g.xt_out && !g.xt_gamma) ||
      (g.epi != EPI_QKV && g.epi != EPI_RESID && g.epi != EPI_GELU && g.epi != EPI_KV))
    return cudaErrorInvalidValue;
  const size_t smem = linear_wide_smem_bytes(g.BN);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  void (*fn)(CUtensorMap, CUtensorMap, LinArgs) =
      g.epi == EPI_QKV ? k_linear_wide<EPI_QKV>
                       : (g.epi == EPI_RESID ? k_linear_wide<EPI_RESID>
                                             : (g.epi == EPI_GELU ? k_linear_wide<EPI_GELU> : k_linear_wide<EPI_KV>));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kWideThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, *tmA, *tmB, g);
}
