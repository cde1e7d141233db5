// Fused linear layer of the action expert on tcgen05, with split-K inside a
// thread-block cluster.
//
// y[t][n] = sum_k W[n][k] X[t][k] for one weight tile of 128 output rows and
// one token tile of BN tokens.  The K range is split over the C CTAs of a
// thread-block cluster (grid.z = C = cluster size); each CTA accumulates its
// slice in TMEM and writes the fp32 tile to a per-rank exchange buffer in
// global memory (L2); after a cluster barrier CTA `rank` sums rows
// [rank*128/C, (rank+1)*128/C) of all C tiles from that buffer (fixed order:
// deterministic) and applies the epilogue:
//   EPI_QKV   scatter to q [B][n_q][H][d_h], k_s [B][n_kv][H][d_h] and
//             v_s^T [B][n_kv][d_h][Hp] (bf16) for the attention kernel;
//   EPI_RESID h[t][n] += y, and per-(128-row block, token) sums of squares of
//             the new h for the next modulated RMSNorm (the cluster combines
//             its ranks' partial sums, rank 0 writes them; or every rank
//             writes its own slot);
//   EPI_GELU  g[t][n] = bf16(GeLU(y)).
// The B operand (tokens) is either TMA-loaded from an activation tensor
// (bmode 0) or built in shared memory from the fp32 residual stream as the
// time-modulated RMSNorm  h / rms(h) * (1 + gamma) + beta  (bmode 1): one
// TMA brings the CTA's h tile while the threads fetch the sums of squares
// and the modulation slices in parallel.  Bmode 2 factors the norm out of
// the product, W u = r W((1 + gamma) h) + W beta: the B operand is the bf16
// (1 + gamma) h that the previous residual epilogue wrote (bmode 2 on
// EPI_RESID), and the QKV / GeLU epilogues apply the row scale r and add
// W beta.
// Packed ternary weights (amode 1 and 2, the W2A8 variant): the 2-bit codes
// arrive by TMA (a ring of stages, or with amode 2 every k-block of the CTA
// at once) and two decoder warps expand them to the bf16 tile the MMA reads.
//
// The weights do not depend on the previous kernel, so their TMA loads are
// issued before griddepcontrol.wait: under programmatic dependent launch the
// weight stream of this layer overlaps the tail of the previous kernel.
//
// Sources: "vla.cpp: A Unified Inference Runtime for Vision-Language-Action
// Models", §III-A Eq. (1) (the velocity network evaluated per Euler step)
// and §III-B Eq. (2) (queries, action keys and values for joint attention).
#include "vla_common.cuh"

namespace {

constexpr uint32_t kA = 128 * 128;  // bytes of one 128 x 64 bf16 weight stage
constexpr int kMaxC = 16;           // largest cluster
constexpr int kPre = 2;             // residual quads prefetched per thread
constexpr int kSlotRound = 32;      // sums-of-squares slots loaded per round (factored norm)
constexpr int kMaxSlots = 256;      // slots a factored-norm map may read (16 ranks x 16 row blocks)
constexpr int kMaxResident = 16;    // k-blocks whose packed codes a CTA holds at once (amode 2)


struct LinSmem {
  uint32_t a, b, hs, pk, region, bars, slot, rstat, gam, bet, wss, total;
};
constexpr uint32_t kPk = 128 * 16;  // one stage of packed ternary codes: 128 rows x 64 codes

__host__ __device__ __forceinline__ LinSmem lin_layout(const LinArgs& g) {
  LinSmem s;
  const uint32_t b_tile = (uint32_t)g.BN * 128u;
  const uint32_t nkb = (uint32_t)(g.KS / 64);
  s.a = 0;
  s.b = (uint32_t)g.stages * kA;
  s.hs = s.b + (g.bmode != 1 ? (uint32_t)g.stages * b_tile : nkb * b_tile);
  s.pk = s.hs + (g.bmode == 1 ? nkb * (uint32_t)g.BN * 256u : 0u);
  // packed codes: a ring of `stages` (amode 1) or every k-block of the CTA (amode 2)
  const uint32_t end = s.pk + (g.amode == 1 ? (uint32_t)g.stages * kPk : (g.amode == 2 ? nkb * kPk : 0u));
  s.region = end;
  s.bars = s.region;                                  // full, empty, done, hbar, aready (+ spare)
  s.slot = s.bars + (4u * (uint32_t)g.stages + 2u) * 8u;
  s.rstat = s.slot + 16u;                             // [BN] (also the epilogue's per-token sums)
  s.gam = s.rstat + (uint32_t)g.BN * 4u;              // [KS]
  s.bet = s.gam + (uint32_t)g.KS * 4u;                // [KS]
  s.wss = s.bet + (uint32_t)g.KS * 4u;                // [4][BN] per-warp sums of squares (C == 1)
  s.total = s.wss + 4u * (uint32_t)g.BN * 4u;
  return s;
}

template <int EPI, int AMODE, int BMODE, int CS>
__global__ void __launch_bounds__(128, 1)
    k_linear(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmH, const LinArgs g) {
  // EPI, AMODE (1: packed ternary weights, W2A8 scaling), BMODE and the
  // cluster size CS (1: no split) are compile-time so that every
  // instantiation carries only its own path: these CTAs run their code once,
  // and instruction fetch is a large part of their time.
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const LinSmem Ls = lin_layout(g);
  const int BN = g.BN, NS = g.stages;
  const int nkb = g.KS / 64;
  const uint32_t b_tile = (uint32_t)BN * 128u;
  uint8_t* Abase = smem + Ls.a;
  uint8_t* Bbase = smem + Ls.b;
  float* Hs = (float*)(smem + Ls.hs);
  uint8_t* Pk = smem + Ls.pk;
  uint64_t* full = (uint64_t*)(smem + Ls.bars);
  uint64_t* empty = full + NS;
  uint64_t* done = empty + NS;
  uint64_t* hbar = done + 1;
  uint64_t* aready = hbar + 1;  // [NS]: decoded ternary A tile and its B tile ready (amode 1)
  uint32_t* tmem_slot = (uint32_t*)(smem + Ls.slot);
  float* rstat = (float*)(smem + Ls.rstat);
  float* gam = (float*)(smem + Ls.gam);
  float* bet = (float*)(smem + Ls.bet);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128;
  const int t0 = blockIdx.y * BN;
  constexpr bool SPLIT = CS > 1;
  constexpr int C = CS;
  const int rank = blockIdx.z;
  const int k0 = rank * g.KS;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)BN) ncols <<= 1;
  VLA_TL(g.tl, 0, 0);

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(hbar, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&aready[s], 3);  // two decoder warps + the producer's B-tile transaction
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(BMODE != 1 ? (const void*)&tmB : (const void*)&tmH);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  VLA_TL(g.tl, 0, 1);

  // Weight prefetch: independent of every earlier kernel.
  const int pre = nkb < NS ? nkb : NS;
  // full[s] carries the A stage (and, for bf16 weights with TMA'd tokens, the
  // B stage); packed ternary stages put their B tile on aready[s] (with the
  // decoders' arrivals) instead, so the codes can be decoded before the
  // previous kernel has finished.
  const uint32_t stage_tx = AMODE == 1 ? kPk : kA + (BMODE != 1 ? b_tile : 0u);
  // A stage i: bf16 tile by TMA, or its 2-bit codes (16 bytes per row per 64 K)
  auto load_a = [&](int i, int s, uint64_t pol) {
    if (AMODE == 1)
      tma_load_2d_hint(Pk + (size_t)s * kPk, &tmA, &full[s], (k0 + i * 64) / 4, g.a_row0 + m0, pol);
    else
      tma_load_2d_hint(Abase + (size_t)s * kA, &tmA, &full[s], k0 + i * 64, g.a_row0 + m0, pol);
  };
  if (warp == 0 && lane == 0) {
    const uint64_t pol = l2_policy_evict_first();
    if (AMODE == 2) {
      // every k-block's codes at once (one barrier): the decode is then
      // paced by the decoders and the MMAs, not by a load per stage
      mbar_arrive_expect_tx(&full[0], (uint32_t)nkb * kPk);
      for (int i = 0; i < nkb; ++i)
        tma_load_2d_hint(Pk + (size_t)i * kPk, &tmA, &full[0], (k0 + i * 64) / 4, g.a_row0 + m0, pol);
    } else {
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], stage_tx);
        load_a(i, i, pol);
      }
    }
  }
  if (threadIdx.x == 0) griddep_launch_dependents();
  const bool decoder = AMODE >= 1 && warp >= 2;
  if (decoder) {
    // Warps 2-3: decode each stage's 2-bit codes (code q+1, little-endian
    // fields) into the bf16 A tile with the 128-byte swizzle the MMA reads.
    // Weights only: this starts before griddepcontrol.wait.
    const int dt = threadIdx.x - 64;
    bool okd = AMODE != 2 || mbar_wait(&full[0], 0, g.status);  // amode 2: every k-block's codes
    if (!okd) s_fail = 1;
    for (int i = 0; okd && i < nkb; ++i) {
      const int s = i % NS;
      // amode 1: stage s's codes have landed; amode 2: the MMAs have
      // released decoded stage s (a stage's first use needs no wait)
      const bool oks = AMODE == 2 ? (i < NS || mbar_wait(&empty[s], ((i / NS) & 1) ^ 1, g.status))
                                  : mbar_wait(&full[s], (i / NS) & 1, g.status);
      if (!oks) {
        s_fail = 1;
        break;
      }
      const uint8_t* pk = Pk + (size_t)(AMODE == 2 ? i : s) * kPk;
      const uint32_t at = smem_u32(Abase + (size_t)s * kA);
      // Rows dt and dt + 64: one 16-byte load of 64 codes each, eight
      // 16-byte chunks out (consecutive lanes cover all eight swizzle phases).
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = dt + h * 64;
        const uint4 cw = *(const uint4*)(pk + r * 16);
        const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {  // codes of k = 8ch .. 8ch+7
          const uint32_t two = (wd[ch >> 1] >> ((ch & 1) * 16)) & 0xFFFFu;
          const uint2 lo = ternary_quad_bf16(two & 0xFFu), hi = ternary_quad_bf16(two >> 8);
          st_shared_v4_u32(at + sw128_offset((uint32_t)r, (uint32_t)ch), make_uint4(lo.x, lo.y, hi.x, hi.y));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aready[s]);
    }
  } else {
    griddep_wait();
  }
  VLA_TL(g.tl, 0, 2);

  int issued = pre;
  if (warp == 0 && lane == 0) {
    if (BMODE == 1) {
      mbar_arrive_expect_tx(hbar, (uint32_t)nkb * (uint32_t)BN * 256u);
      for (int i = 0; i < nkb; ++i) tma_load_2d(Hs + (size_t)i * BN * 64, &tmH, hbar, k0 + i * 64, t0);
    } else if (AMODE >= 1) {
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&aready[i], b_tile);
        tma_load_2d(Bbase + (size_t)i * b_tile, &tmB, &aready[i], k0 + i * 64, t0);
      }
    } else {
      for (int i = 0; i < pre; ++i) tma_load_2d(Bbase + (size_t)i * b_tile, &tmB, &full[i], k0 + i * 64, t0);
    }
  }
  if (BMODE == 1) {
    // All four warps: B slice = modulated RMSNorm of h over this rank's K
    // range.  Thread tid always handles the same 8-column chunk kc (so its
    // gamma / beta stay in registers) for tokens t = tid / kcs + j * (128 / kcs).
    const int tid = threadIdx.x;
    for (int t = tid; t < BN; t += 128) {
      const int tt = t0 + t;
      float r = 0.f;
      if (tt < g.T) {
        float v[kMaxC];
#pragma unroll
        for (int s = 0; s < kMaxC; ++s) v[s] = s < g.n_ss_in ? g.ss_in[(size_t)s * g.T + tt] : 0.f;
        float ss = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxC; ++s) ss += v[s];
        r = rsqrtf(ss / (float)g.D + g.eps);
      }
      rstat[t] = r;
    }
    const int kcs = g.KS / 8;  // 8-column chunks per token (divides 128: KS <= 1024, power of two)
    const int kc = tid % kcs;
    const int tstep = 128 / kcs;
    const float4* gp = (const float4*)(g.gamma + k0 + kc * 8);
    const float4* bp = (const float4*)(g.beta + k0 + kc * 8);
    const float4 g0 = gp[0], g1 = gp[1], b0 = bp[0], b1 = bp[1];
    __syncthreads();
    VLA_TL(g.tl, 32, 8);
    if (!mbar_wait(hbar, 0, g.status)) s_fail = 1;
    VLA_TL(g.tl, 32, 9);
    const uint32_t bb = smem_u32(Bbase) + (uint32_t)(kc >> 3) * b_tile;
    const float* hcol = Hs + (size_t)(kc >> 3) * BN * 64 + (kc & 7) * 8;
#pragma unroll 4
    for (int t = tid / kcs; t < BN; t += tstep) {
      const int tt = t0 + t;
      uint4 pk = make_uint4(0u, 0u, 0u, 0u);
      if (tt < g.T) {
        const float r = rstat[t];
        const float4* hp = (const float4*)(hcol + (size_t)t * 64);
        const float4 h0 = hp[0], h1 = hp[1];
        pk.x = pack_bf16x2(h0.x * r * (1.f + g0.x) + b0.x, h0.y * r * (1.f + g0.y) + b0.y);
        pk.y = pack_bf16x2(h0.z * r * (1.f + g0.z) + b0.z, h0.w * r * (1.f + g0.w) + b0.w);
        pk.z = pack_bf16x2(h1.x * r * (1.f + g1.x) + b1.x, h1.y * r * (1.f + g1.y) + b1.y);
        pk.w = pack_bf16x2(h1.z * r * (1.f + g1.z) + b1.z, h1.w * r * (1.f + g1.w) + b1.w);
      }
      st_shared_v4_u32(bb + sw128_offset((uint32_t)t, (uint32_t)(kc & 7)), pk);
    }
    fence_proxy_async_smem();
    __syncthreads();
    VLA_TL(g.tl, 32, 10);
  }
  if (warp == 0 && lane == 0) {
    const uint64_t pol = l2_policy_evict_first();
    for (int i = pre; i < nkb; ++i) {
      const int s = i % NS;
      if (!mbar_wait(&empty[s], ((i / NS) & 1) ^ 1, g.status)) {
        s_fail = 1;
        break;
      }
      if (AMODE != 2) {
        mbar_arrive_expect_tx(&full[s], stage_tx);
        load_a(i, s, pol);
      }
      if (AMODE >= 1) {
        mbar_arrive_expect_tx(&aready[s], b_tile);
        tma_load_2d(Bbase + (size_t)s * b_tile, &tmB, &aready[s], k0 + i * 64, t0);
      } else if (BMODE != 1) {
        tma_load_2d(Bbase + (size_t)s * b_tile, &tmB, &full[s], k0 + i * 64, t0);
      }
      issued = i + 1;
    }
  }
  if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, BN);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % NS;
      // One wait per stage: the TMA transaction of the stage (bf16 weights),
      // or the decoded tile plus its B tile (packed ternary weights).
      if (s_fail || !mbar_wait(AMODE >= 1 ? &aready[s] : &full[s], (i / NS) & 1, g.status)) {
        s_fail = 1;
        break;
      }
      if (i == 0) VLA_TL(g.tl, 32, 3);
      if (i == 1) VLA_TL(g.tl, 32, 12);
      if (i == 2) VLA_TL(g.tl, 32, 13);
      if (i == 3) VLA_TL(g.tl, 32, 14);
      if (i == nkb - 1) VLA_TL(g.tl, 32, 15);
      tc_fence_after();
      const uint32_t a_addr = smem_u32(Abase + (size_t)s * kA);
      const uint32_t b_addr = smem_u32(Bbase + (size_t)(BMODE != 1 ? s : i) * b_tile);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_bf16(tmem, sdesc_k128(a_addr + k * 32), sdesc_k128(b_addr + k * 32), idesc, (i > 0 || k > 0) ? 1u : 0u);
      if (i + NS < nkb) umma_commit(&empty[s]);  // only a stage that will be refilled needs releasing
    }
    umma_commit(done);
    VLA_TL(g.tl, 32, 4);
  }
  __syncwarp();
  if (decoder) griddep_wait();  // the epilogue reads and writes activations

  // Epilogue geometry: rank r owns rows [r*RPR, (r+1)*RPR) of the tile.
  const int RPR = 128 / C;
  const int qpc = RPR / 4;  // float4 quads per token column
  const int nquads = qpc * BN;
  const int iters = (nquads + 127) / 128;
  // Prefetch the residual rows this thread will update (independent of the MMA).
  float4 hpre[kPre];
  if (EPI == EPI_RESID) {
#pragma unroll
    for (int it = 0; it < kPre; ++it) {
      const int f = threadIdx.x + it * 128;
      hpre[it] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (it < iters && f < nquads) {
        const int col = f / qpc, quad = f - col * qpc;
        const int n = m0 + rank * RPR + quad * 4, t = t0 + col;
        if (t < g.T && n < g.N) hpre[it] = *(const float4*)(g.h + (size_t)t * g.D + n);
      }
    }
  }

  // Factored modulated norm (BMODE 2), fetched while the MMAs run: the row
  // scales r_t of this tile's tokens into rstat (QKV / GeLU maps), and the
  // thread's W beta values (QKV / GeLU) or next-norm scales 1 + gamma
  // (residual map, which writes (1 + gamma) h_new for the next normed map).
  // Split path: the thread's rows are the same quad in every iteration.
  constexpr bool FN_IN = BMODE == 2 && (EPI == EPI_QKV || EPI == EPI_GELU);
  constexpr bool FN_OUT = BMODE == 2 && EPI == EPI_RESID;
  float4 fn4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (FN_IN && threadIdx.x >= 64) {  // warps 2-3 (the producer and MMA threads are still busy)
    for (int t = threadIdx.x - 64; t < BN; t += 64) {
      float ssum = 0.f;
      for (int s0 = 0; s0 < g.fn_nss; s0 += kSlotRound) {
        float v[kSlotRound];  // a round of slot loads in flight at once; fixed summation order
#pragma unroll
        for (int sl = 0; sl < kSlotRound; ++sl)
          v[sl] = (s0 + sl < g.fn_nss && t0 + t < g.T) ? g.fn_ss[(size_t)(s0 + sl) * g.T + t0 + t] : 0.f;
#pragma unroll
        for (int sl = 0; sl < kSlotRound; ++sl) ssum += v[sl];
      }
      rstat[t] = rsqrtf(ssum / (float)g.D + g.eps);
    }
  }
  if (FN_IN || FN_OUT) {
    const float* src = FN_IN ? g.fn_c : g.xt_gamma;
    const float add = FN_IN ? 0.f : 1.f;
    if (SPLIT) {
      const int n = m0 + rank * RPR + (threadIdx.x % qpc) * 4;
      if (n < g.N) {
        fn4 = *(const float4*)(src + n);
        fn4.x += add; fn4.y += add; fn4.z += add; fn4.w += add;
      }
    } else {
      const int n = m0 + threadIdx.x;
      if (n < g.N) fn4.x = src[n] + add;
    }
  }
  // W2A8 scales, fetched while the MMAs run: the thread's weight-scale quad
  // (the same rows in every epilogue iteration of the split path, since its
  // quads per column divide 128) and the token scales of its first two
  // iterations.
  float4 be_pre = make_float4(0.f, 0.f, 0.f, 0.f);
  float al_pre[2] = {0.f, 0.f};
  if (AMODE >= 1 && SPLIT) {
    const int quad = threadIdx.x % qpc;
    const int n = m0 + rank * RPR + quad * 4;
    if (n < g.N)
      be_pre = g.wbeta ? *(const float4*)(g.wbeta + (size_t)g.layer * g.beta_stride + g.beta_off + n)
                       : make_float4(g.beta_val, g.beta_val, g.beta_val, g.beta_val);
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int t = t0 + (threadIdx.x + it * 128) / qpc;
      if (it < iters && t < g.T) al_pre[it] = g.alpha[t];
    }
  }

  if (!mbar_wait(done, 0, g.status)) s_fail = 1;
  tc_fence_after();
  __syncthreads();
  VLA_TL(g.tl, 0, 5);
  const bool ok = (s_fail == 0);
  const int tile = blockIdx.y * gridDim.x + blockIdx.x;
  const int tcols = (g.T - t0) < BN ? (g.T - t0) : BN;  // valid token columns

  if (!SPLIT) {
    // No split: every thread owns one output row n and applies the epilogue
    // straight from TMEM (lanes hold consecutive rows: coalesced stores).
    const int row = warp * 32 + lane;
    const int n = m0 + row;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    float* wss = (float*)(smem + Ls.wss);
    int slot = 0;
    if (EPI == EPI_QKV) slot = n < g.qdim ? 0 : (n < g.qdim + g.kvdim ? 1 : 2);
    const float be = (AMODE >= 1 && n < g.N)
                         ? (g.wbeta ? g.wbeta[(size_t)g.layer * g.beta_stride + g.beta_off + n] : g.beta_val)
                         : 0.f;
    for (int c0 = 0; c0 < tcols; c0 += 16) {
      float v[16];
      if (ok) {
        tmem_ld16(taddr + (uint32_t)c0, v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = t0 + c0 + j;
        const bool valid = ok && c0 + j < tcols && n < g.N;
        float y = v[j];
        if (AMODE >= 1 && valid) {
          if (EPI != EPI_W2A8_OUT && g.accout) g.accout[(size_t)t * g.N + n] = (int32_t)y;  // diagnostic tap
          y = w2a8_scale(y, g.alpha[t], be);
        }
        if (FN_IN) y = fmaf(rstat[c0 + j], y, fn4.x);
        float sq = 0.f;
        if (valid) {
          if (EPI == EPI_RESID) {
            float* hp = g.h + (size_t)t * g.D + n;
            const float hv = *hp + y;
            *hp = hv;
            if (FN_OUT) g.xt_out[(size_t)t * g.D + n] = __float2bfloat16_rn(fn4.x * hv);
            sq = hv * hv;
          } else if (EPI == EPI_GELU) {
            if (g.g32)
              g.g32[(size_t)t * g.ldg + n] = gelu_exact(y);
            else
              g.g[(size_t)t * g.ldg + n] = __float2bfloat16_rn(gelu_exact(y));
          } else if (EPI == EPI_W2A8_OUT) {
            g.yout[(size_t)t * g.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
            if (g.accout) g.accout[(size_t)t * g.N + n] = (int32_t)v[j];
          } else if (EPI == EPI_KV) {
            // prefix cache (Eq. 2): row n = [layer][K | V][kv head][d], token t = [b][p]
            const int kl = n / (2 * g.kvdim), rem = n - kl * 2 * g.kvdim, kw = rem / g.kvdim;
            const int r2 = rem - kw * g.kvdim, gk = r2 / g.d_h, d = r2 - gk * g.d_h;
            const int b = t / g.kv_P, p = t - b * g.kv_P;
            const size_t head = ((size_t)kl * g.kv_B + b) * g.n_kv + gk;
            if (kw == 0)
              g.kc_out[(head * g.kv_P + p) * g.d_h + d] = __float2bfloat16_rn(y);
            else
              g.vc_out[(head * g.d_h + d) * g.kv_P8 + p] = __float2bfloat16_rn(y);
          } else {  // EPI_QKV
            const int b = t / g.H, i = t - b * g.H;
            const bf16 bv = __float2bfloat16_rn(y);
            if (slot == 0) {
              const int jh = n / g.d_h, d = n - jh * g.d_h;
              g.q[(((size_t)b * g.n_q + jh) * g.H + i) * g.d_h + d] = bv;
            } else if (slot == 1) {
              const int r = n - g.qdim, gk = r / g.d_h, d = r - gk * g.d_h;
              g.ks[(((size_t)b * g.n_kv + gk) * g.H + i) * g.d_h + d] = bv;
            } else {
              const int r = n - g.qdim - g.kvdim, gk = r / g.d_h, d = r - gk * g.d_h;
              g.vst[(((size_t)b * g.n_kv + gk) * g.d_h + d) * g.Hp + i] = bv;
            }
          }
        }
        if (EPI == EPI_RESID) {
          sq = warp_sum(sq);
          if (lane == 0) wss[warp * BN + c0 + j] = sq;
        }
      }
    }
    if (EPI == EPI_RESID && g.ss_out) {
      __syncthreads();
      for (int col = threadIdx.x; col < tcols; col += 128)
        g.ss_out[(size_t)blockIdx.x * g.T + t0 + col] =
            wss[col] + wss[BN + col] + wss[2 * BN + col] + wss[3 * BN + col];
    }
  } else {
  // Publish the fp32 partial tile through L2, column-major [col][row]
  // (padding token columns are skipped).
  float* mypart = g.xpart + ((size_t)tile * C + rank) * (size_t)BN * 128;
  if (ok) {
    const int row = warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c0 = 0; c0 < tcols; c0 += 64) {  // up to 64 columns per TMEM wait
      uint32_t r[64];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c0 + q * 16 < tcols) tmem_ld16_nowait(taddr + (uint32_t)(c0 + q * 16), r + q * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c0 + q * 16 < tcols) tmem_wait16(r + q * 16);
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (c0 + j < tcols) __stcg(mypart + (size_t)(c0 + j) * 128 + row, __uint_as_float(r[j]));
    }
  }
  cluster_sync_all();
  VLA_TL(g.tl, 0, 6);

  // Cluster reduction (fixed rank order) and epilogue.  The partial sums of
  // the first kPre iterations are gathered together so their L2 loads overlap.
  const float* tpart = g.xpart + (size_t)tile * C * (size_t)BN * 128;
  auto geom = [&](int it, bool& live, int& col, int& quad) {
    const int f = threadIdx.x + it * 128;
    live = ok && f < nquads && f / qpc < tcols;
    col = live ? f / qpc : 0;
    quad = live ? f - col * qpc : 0;
  };
  auto epilogue = [&](float4 acc, bool live, int col, int quad, float4 hprev, bool have_prev, int it) {
    const int rloc = rank * RPR + quad * 4;
    const int n = m0 + rloc, t = t0 + col;
    const bool valid = live && t < g.T && n < g.N;
    const float4 raw = acc;
    if (AMODE >= 1 && valid) {
      // Eq. (4): exact integer accumulators scaled to bf16
      const float al = it < 2 ? al_pre[it] : g.alpha[t];
      const float4 be = be_pre;
      acc.x = w2a8_scale(acc.x, al, be.x);
      acc.y = w2a8_scale(acc.y, al, be.y);
      acc.z = w2a8_scale(acc.z, al, be.z);
      acc.w = w2a8_scale(acc.w, al, be.w);
      if (EPI != EPI_W2A8_OUT && g.accout)  // diagnostic tap of the exact accumulators
        *(int4*)(g.accout + (size_t)t * g.N + n) = make_int4((int)raw.x, (int)raw.y, (int)raw.z, (int)raw.w);
    }
    if (FN_IN && valid) {
      const float rr = rstat[col];
      acc.x = fmaf(rr, acc.x, fn4.x);
      acc.y = fmaf(rr, acc.y, fn4.y);
      acc.z = fmaf(rr, acc.z, fn4.z);
      acc.w = fmaf(rr, acc.w, fn4.w);
    }
    if (EPI == EPI_RESID) {
      float ss = 0.f;
      if (valid) {
        float4* hp = (float4*)(g.h + (size_t)t * g.D + n);
        float4 hv = have_prev ? hprev : *hp;
        hv.x += acc.x; hv.y += acc.y; hv.z += acc.z; hv.w += acc.w;
        *hp = hv;
        if (FN_OUT) {
          uint2 xk;
          xk.x = pack_bf16x2(fn4.x * hv.x, fn4.y * hv.y);
          xk.y = pack_bf16x2(fn4.z * hv.z, fn4.w * hv.w);
          *(uint2*)(g.xt_out + (size_t)t * g.D + n) = xk;
        }
        ss = hv.x * hv.x + hv.y * hv.y + hv.z * hv.z + hv.w * hv.w;
      }
      for (int o = qpc >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (live && quad == 0) rstat[col] = ss;
    } else if (EPI == EPI_GELU) {
      if (valid) {
        if (g.g32) {
          *(float4*)(g.g32 + (size_t)t * g.ldg + n) =
              make_float4(gelu_exact(acc.x), gelu_exact(acc.y), gelu_exact(acc.z), gelu_exact(acc.w));
        } else {
          uint2 pk;
          pk.x = pack_bf16x2(gelu_exact(acc.x), gelu_exact(acc.y));
          pk.y = pack_bf16x2(gelu_exact(acc.z), gelu_exact(acc.w));
          *(uint2*)(g.g + (size_t)t * g.ldg + n) = pk;
        }
      }
    } else if (EPI == EPI_W2A8_OUT) {
      if (valid) {
        uint2 pk;
        pk.x = pack_bf16x2(acc.x, acc.y);
        pk.y = pack_bf16x2(acc.z, acc.w);
        *(uint2*)(g.yout + (size_t)t * g.N + n) = pk;
        if (g.accout)
          *(int4*)(g.accout + (size_t)t * g.N + n) = make_int4((int)raw.x, (int)raw.y, (int)raw.z, (int)raw.w);
      }
    } else {  // EPI_QKV: a 4-row quad lies inside one head of q, k or v
      if (valid) {
        const int b = t / g.H, i = t - b * g.H;
        if (n < g.qdim + g.kvdim) {
          const bool isq = n < g.qdim;
          const int r = isq ? n : n - g.qdim;
          const int j = r / g.d_h, d = r - j * g.d_h;
          bf16* dst = isq ? g.q + (((size_t)b * g.n_q + j) * g.H + i) * g.d_h + d
                          : g.ks + (((size_t)b * g.n_kv + j) * g.H + i) * g.d_h + d;
          uint2 pk;
          pk.x = pack_bf16x2(acc.x, acc.y);
          pk.y = pack_bf16x2(acc.z, acc.w);
          *(uint2*)dst = pk;
        } else {
          const int r = n - g.qdim - g.kvdim;
          const int gk = r / g.d_h, d = r - gk * g.d_h;
          bf16* dst = g.vst + (((size_t)b * g.n_kv + gk) * g.d_h + d) * g.Hp + i;
          dst[0] = __float2bfloat16_rn(acc.x);
          dst[g.Hp] = __float2bfloat16_rn(acc.y);
          dst[2 * g.Hp] = __float2bfloat16_rn(acc.z);
          dst[3 * g.Hp] = __float2bfloat16_rn(acc.w);
        }
      }
    }
  };
  {
    // Iterations 0 and 1 (the only ones at small token counts): issue every
    // partial load first, then sum, so the loads overlap.
    bool lv0, lv1;
    int cl0, qd0, cl1, qd1;
    geom(0, lv0, cl0, qd0);
    geom(1, lv1, cl1, qd1);
    if (iters < 1) lv0 = false;
    if (iters < 2) lv1 = false;
    const float* p0 = tpart + (size_t)cl0 * 128 + rank * RPR + qd0 * 4;
    const float* p1 = tpart + (size_t)cl1 * 128 + rank * RPR + qd1 * 4;
    float4 v0[C], v1[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      v0[c] = lv0 ? __ldcg((const float4*)(p0 + (size_t)c * BN * 128)) : make_float4(0.f, 0.f, 0.f, 0.f);
      v1[c] = lv1 ? __ldcg((const float4*)(p1 + (size_t)c * BN * 128)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      a0.x += v0[c].x; a0.y += v0[c].y; a0.z += v0[c].z; a0.w += v0[c].w;
      a1.x += v1[c].x; a1.y += v1[c].y; a1.z += v1[c].z; a1.w += v1[c].w;
    }
    if (iters >= 1) epilogue(a0, lv0, cl0, qd0, hpre[0], EPI == EPI_RESID, 0);
    if (iters >= 2) epilogue(a1, lv1, cl1, qd1, hpre[1], EPI == EPI_RESID, 1);
  }
  for (int it = 2; it < iters; ++it) {
    bool live;
    int col, quad;
    geom(it, live, col, quad);
    float4 v[C];
#pragma unroll
    for (int c = 0; c < C; ++c)
      v[c] = live ? __ldcg((const float4*)(tpart + (size_t)c * BN * 128 + (size_t)col * 128 + rank * RPR +
                                                      quad * 4))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < C; ++c) {
      acc.x += v[c].x; acc.y += v[c].y; acc.z += v[c].z; acc.w += v[c].w;
    }
    epilogue(acc, live, col, quad, make_float4(0.f, 0.f, 0.f, 0.f), false, it);
  }
  VLA_TL(g.tl, 0, 11);
  if (EPI == EPI_RESID && g.ss_out && g.ss_per_rank) {
    // Each rank's own slot; the consumer sums them.
    __syncthreads();
    if (ok)
      for (int col = threadIdx.x; col < tcols; col += 128)
        g.ss_out[((size_t)blockIdx.x * C + rank) * g.T + t0 + col] = rstat[col];
  } else if (EPI == EPI_RESID && g.ss_out) {
    // Rank 0 combines the ranks' per-token sums of squares (fixed order).
    __syncthreads();
    float* myss = g.xss + ((size_t)tile * C + rank) * BN;
    for (int col = threadIdx.x; col < tcols; col += 128) __stcg(myss + col, rstat[col]);
    cluster_sync_all();
    if (rank == 0 && ok) {
      const float* tss = g.xss + (size_t)tile * C * BN;
      for (int col = threadIdx.x; col < tcols; col += 128) {
        float v[C];
#pragma unroll
        for (int c = 0; c < C; ++c) v[c] = __ldcg(tss + (size_t)c * BN + col);
        float s2 = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) s2 += v[c];
        g.ss_out[(size_t)blockIdx.x * g.T + t0 + col] = s2;
      }
    }
  }
  }  // C > 1

  // Drain own TMA copies (only relevant after a timeout) and free TMEM.
  if (warp == 0 && lane == 0) {
    const int first = issued > NS ? issued - NS : 0;
    for (int i = first; i < issued; ++i) {
      if (AMODE != 2) mbar_drain(&full[i % NS], (i / NS) & 1);
      if (AMODE >= 1) mbar_drain(&aready[i % NS], (i / NS) & 1);
    }
    if (AMODE == 2) mbar_drain(&full[0], 0);
    if (BMODE == 1) mbar_drain(hbar, 0);
    mbar_drain(done, 0);  // the MMA warp always commits `done`
  }
  tc_fence_before();
  __syncthreads();
  VLA_TL(g.tl, 0, 7);
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

}  // namespace

size_t linear_smem_bytes(const LinArgs& g) { return 1024 + lin_layout(g).total; }

template <int EPI, int AMODE, int BMODE>
cudaError_t init_one() {
  cudaError_t e = set_max_dyn_smem(k_linear<EPI, AMODE, BMODE, 1>);
#define VLA_LIN_INIT(CSZ)                                                                                   \
  if (e == cudaSuccess) e = set_max_dyn_smem(k_linear<EPI, AMODE, BMODE, CSZ>);                          \
  if (e == cudaSuccess)                                                                                   \
    e = cudaFuncSetAttribute(k_linear<EPI, AMODE, BMODE, CSZ>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  VLA_LIN_INIT(2)
  VLA_LIN_INIT(4)
  VLA_LIN_INIT(8)
  VLA_LIN_INIT(16)
#undef VLA_LIN_INIT
  return e;
}

cudaError_t linear_kernels_init() {
  cudaError_t e = cudaSuccess;
  // bf16 weights: every epilogue with TMA'd or norm-built tokens
  if (e == cudaSuccess) e = init_one<EPI_QKV, 0, 0>();
  if (e == cudaSuccess) e = init_one<EPI_QKV, 0, 1>();
  if (e == cudaSuccess) e = init_one<EPI_RESID, 0, 0>();
  if (e == cudaSuccess) e = init_one<EPI_GELU, 0, 0>();
  if (e == cudaSuccess) e = init_one<EPI_GELU, 0, 1>();
  // factored modulated norm (bmode 2)
  if (e == cudaSuccess) e = init_one<EPI_QKV, 0, 2>();
  if (e == cudaSuccess) e = init_one<EPI_RESID, 0, 2>();
  if (e == cudaSuccess) e = init_one<EPI_GELU, 0, 2>();
  // packed ternary weights (W2A8)
  if (e == cudaSuccess) e = init_one<EPI_QKV, 1, 0>();
  if (e == cudaSuccess) e = init_one<EPI_RESID, 1, 0>();
  if (e == cudaSuccess) e = init_one<EPI_GELU, 1, 0>();
  if (e == cudaSuccess) e = init_one<EPI_W2A8_OUT, 1, 0>();
  // packed ternary weights, every k-block's codes resident
  if (e == cudaSuccess) e = init_one<EPI_QKV, 2, 0>();
  if (e == cudaSuccess) e = init_one<EPI_RESID, 2, 0>();
  if (e == cudaSuccess) e = init_one<EPI_GELU, 2, 0>();
  if (e == cudaSuccess) e = init_one<EPI_W2A8_OUT, 2, 0>();
  if (e == cudaSuccess) e = set_max_dyn_smem(k_linear<EPI_KV, 1, 0, 1>);
  return e;
}

cudaError_t launch_linear(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmH, const LinArgs& g,
                          int tiles_n, int tiles_t, int C, cudaStream_t st) {
  if (g.BN < 16 || g.BN > 256 || g.BN % 16 || g.KS % 64 || g.KS < 64 || g.stages < 1 || C < 1 || C > kMaxC ||
      (C & (C - 1)) || g.N % 4 || (g.bmode == 1 && (g.n_ss_in < 1 || g.n_ss_in > kMaxC)) ||
      (g.amode >= 1 && g.bmode != 0) || (g.amode >= 1) != (g.w2a8 == 1) || g.amode > 2 ||
      (g.amode == 2 && g.KS / 64 > kMaxResident) ||
      (g.bmode == 2 && g.epi == EPI_RESID && (!g.xt_out || !g.xt_gamma)) ||
      (g.bmode == 2 && (g.epi == EPI_QKV || g.epi == EPI_GELU) &&
       (!g.fn_c || !g.fn_ss || g.fn_nss < 1 || g.fn_nss > kMaxSlots)))
    return cudaErrorInvalidValue;
  const size_t smem = linear_smem_bytes(g);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  void (*fn)(CUtensorMap, CUtensorMap, CUtensorMap, LinArgs) = nullptr;
#define VLA_LIN_CASE(E, A, B)                                                                             \
  if (g.epi == E && g.amode == A && g.bmode == B)                                                        \
    fn = C == 16 ? k_linear<E, A, B, 16>                                                                 \
                 : (C == 8 ? k_linear<E, A, B, 8> : (C == 4 ? k_linear<E, A, B, 4> : (C == 2 ? k_linear<E, A, B, 2> : k_linear<E, A, B, 1>)));
  VLA_LIN_CASE(EPI_QKV, 0, 0)
  VLA_LIN_CASE(EPI_QKV, 0, 1)
  VLA_LIN_CASE(EPI_RESID, 0, 0)
  VLA_LIN_CASE(EPI_GELU, 0, 0)
  VLA_LIN_CASE(EPI_GELU, 0, 1)
  VLA_LIN_CASE(EPI_QKV, 0, 2)
  VLA_LIN_CASE(EPI_RESID, 0, 2)
  VLA_LIN_CASE(EPI_GELU, 0, 2)
  VLA_LIN_CASE(EPI_QKV, 1, 0)
  VLA_LIN_CASE(EPI_RESID, 1, 0)
  VLA_LIN_CASE(EPI_GELU, 1, 0)
  VLA_LIN_CASE(EPI_W2A8_OUT, 1, 0)
  VLA_LIN_CASE(EPI_QKV, 2, 0)
  VLA_LIN_CASE(EPI_RESID, 2, 0)
  VLA_LIN_CASE(EPI_GELU, 2, 0)
  VLA_LIN_CASE(EPI_W2A8_OUT, 2, 0)
#undef VLA_LIN_CASE
  if (g.epi == EPI_KV) fn = (g.amode == 1 && C == 1) ? k_linear<EPI_KV, 1, 0, 1> : nullptr;
  if (!fn) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, tiles_t, C);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = C;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, *tmA, *tmB, *tmH, g);
}
