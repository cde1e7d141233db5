// The whole S-step Euler solve of a few-token request as ONE persistent
// kernel ("vla.cpp: A Unified Inference Runtime for Vision-Language-Action
// Models", §III-A Eq. (1) integrated over the cached prefix of §III-B Eq. (2);
// the solver loop as a single launch of the latency model, Eq. (3)).
//
// At batch 1 the velocity network is bound by its weight bytes: every Euler
// step streams each token-dependent weight once and does little arithmetic
// with it.  A chain of one kernel per linear map pays a launch boundary,
// a first-load latency and a split-K exchange per map, several times the time
// the map's weights take over HBM.  Here one CTA per SM lives for the whole
// solve (cooperative launch, so every CTA is resident) and the work of a layer
// runs as five phases separated by grid-wide barriers:
//   A  [W_q;W_k;W_v] over the modulated-norm input        -> acc_qkv (fp32)
//   B  joint attention per (query tile, 128-key chunk)    -> partial O, (m, l)
//   C  W_o over the merged attention output               -> h += (residual)
//   D  W_up over the modulated-norm input                 -> acc_up (fp32)
//   E  W_down over GeLU(acc_up)                           -> h += (residual)
// and a head phase per step (final norm, W_out, Euler update, and the input
// projection of the next step's chunk).
//
// Weight streaming.  Weights do not depend on activations, so warp 0 streams
// every weight tile this CTA will ever multiply, in consumption order, into a
// ring of 128 x 64 bf16 shared-memory stages, independently of the phases:
// while the CTA waits at a barrier or runs attention, its next phases'
// weights are already arriving.  The work of each linear phase is the list of
// (128-row tile, 64-wide K block) units of its weight matrix, cut into G
// contiguous, equal ranges for the G CTAs, so every SM streams the same
// number of weight bytes.  A CTA's partial sums are added to the fp32 output
// in global memory with reductions (red.global.add), which also performs the
// residual additions of C and E.  (The order of those additions varies from
// run to run, so results agree to fp32 rounding, not bit for bit.)
//
// The modulated RMSNorm is factored out of the GEMM: with
// u = h r (1 + gamma) + beta,  y = W u = r (W ((1 + gamma) h)) + W beta,
// so the B operand is bf16((1 + gamma) h) (no row statistics needed before
// the product), the row scale r = 1 / rms(h) is applied by the consumer of
// the sums, and W beta is a per-(step, layer) vector computed once per handle.
// The rms values are computed during the phase that multiplies (A, D) by the
// CTAs that own one token each, so no extra barrier is needed.
//
// Attention: one work unit per (observation, K/V head, 128-row query tile,
// 128-key chunk of [prefix ; action keys]).  Q and the action keys / values
// are formed from acc_qkv (r acc + W beta, in bf16); cached keys and V^T come
// from the cache by TMA.  S = Q K^T on tcgen05 (d_h / 64 sub-tiles, double
// buffered), softmax in fp32 (one row per thread), P in bf16, O = P V on
// tcgen05; each unit writes its unnormalised O (bf16) with the row maximum m
// and sum l.  Phase C merges the chunks of a row while it builds its B
// operand: o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
//
// Warp roles (256 threads): warp 0 lane 0 streams weights; warp 1 lane 0
// issues the MMAs (and attention TMA loads); warp 2 lane 0 runs the grid
// barrier; warps 1-7 build operands; warps 4-7 run epilogues and the
// softmax (TMEM lane quarter = warp % 4).
#include <math.h>

#include "vla_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWork = 224;            // threads of warps 1..7
constexpr uint32_t kStage = 16384;    // one 128 x 64 bf16 weight tile
constexpr int kKC = 128;              // keys per attention unit
constexpr uint32_t kWorkBytes = 98304;  // operand region (linear B tiles / attention buffers)
constexpr int kBarWork = 1;           // named barrier over warps 1..7

struct PLayout {
  uint32_t ring, work, bars, misc, total;
  int R;
};

__host__ __device__ inline PLayout persist_layout(int D) {
  PLayout s;
  s.work = 0;
  s.bars = kWorkBytes;
  // mbarriers: full[R], empty[R], mma_done, kbar[2], qkfree[2], sdone, vbar, odone (+ pad)
  s.misc = s.bars + 64 * 8;
  // misc: tmem slot, flags, reduction slots, row (m, l) [128], x [d_a <= 64], head row [D]
  const uint32_t misc_bytes = 256 + 128 * 8 + 64 * 4 + (uint32_t)D * 4;
  uint32_t ring0 = (s.misc + misc_bytes + 1023u) & ~1023u;
  const uint32_t budget = 227u * 1024u - 1024u;  // minus the base alignment slack
  int R = (int)((budget - ring0) / kStage);
  if (R > 16) R = 16;
  s.R = R;
  s.ring = ring0;
  s.total = ring0 + (uint32_t)R * kStage;
  return s;
}

// ---------------------------------------------------------------------------
// Small PTX helpers local to this kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const void* map, uint64_t* bar, int x, int y, int z,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg((const float4*)p); }
__device__ __forceinline__ void stcg4(float* p, float4 v) { __stcg((float4*)p, v); }
__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}
__device__ __forceinline__ void unpack8(uint4 w, float* v) {
  const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(a[i] << 16);
    v[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
  }
}

// Sum over the 224 threads of warps 1..7 (`red` holds 8 floats); every
// participating thread gets the result.
__device__ __forceinline__ float work_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) - 1;
  v = warp_sum(v);
  if (lane == 0) red[w] = v;
  named_bar_sync(kBarWork, kWork);
  float r = 0.f;
#pragma unroll
  for (int i = 0; i < 7; ++i) r += red[i];
  named_bar_sync(kBarWork, kWork);
  return r;
}

// Grid-wide barrier over the G persistent CTAs: arrival counter in global
// memory (release), bounded poll (acquire).  Called by the 224 work threads.
__device__ __forceinline__ bool grid_sync(const PersistArgs& a, unsigned target, volatile int* fail) {
  tc_fence_before();
  named_bar_sync(kBarWork, kWork);
  if (threadIdx.x == 64) {
    __threadfence();
    atomicAdd(a.bar, 1u);
    const uint64_t t0 = globaltimer_ns();
    const uint64_t lim = wait_limit_ns(a.status);
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.bar) : "memory");
      if (v >= target) break;
      if (globaltimer_ns() - t0 > lim) {
        latch_error(a.status, VLA_DEV_TIMEOUT);
        *fail = 1;
        break;
      }
      if (*(volatile int*)a.status == VLA_DEV_TIMEOUT) {
        *fail = 1;
        break;
      }
    }
    __threadfence();
  }
  named_bar_sync(kBarWork, kWork);
  tc_fence_after();
  return *fail == 0;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    k_solver_persist(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                     const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmW3,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmVt,
                     const PersistArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const PLayout Ls = persist_layout(a.D);
  const int R = Ls.R;
  uint8_t* work = smem + Ls.work;
  uint8_t* ring = smem + Ls.ring;
  uint64_t* bars = (uint64_t*)(smem + Ls.bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + 16;
  uint64_t* mma_done = bars + 32;
  uint64_t* kbar = bars + 33;    // [2]
  uint64_t* qkfree = bars + 35;  // [2]
  uint64_t* sdone = bars + 37;
  uint64_t* vbar = bars + 38;
  uint64_t* odone = bars + 39;
  uint8_t* misc = smem + Ls.misc;
  uint32_t* tmem_slot = (uint32_t*)misc;
  volatile int* s_fail = (volatile int*)(misc + 16);  // a wait gave up: leave
  volatile int* s_stop = (volatile int*)(misc + 20);  // tells the weight producer to stop
  float* red = (float*)(misc + 32);                   // [8]
  float2* rowml = (float2*)(misc + 256);              // [128] (m, l) of this unit's rows
  float* xs = (float*)(misc + 256 + 128 * 8);         // [64] next chunk of one token
  float* hrow = xs + 64;                              // [D] one token's row (head phase)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int T = a.T, D = a.D, L = a.L, BN = a.BN;

  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kbar[i], 1);
      mbar_init(&qkfree[i], 1);
    }
    mbar_init(sdone, 1);
    mbar_init(vbar, 1);
    mbar_init(odone, 1);
    *s_fail = 0;
    *s_stop = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW0);
    tma_prefetch_desc(&tmW1);
    tma_prefetch_desc(&tmW2);
    tma_prefetch_desc(&tmW3);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Unit range of this CTA in linear phase ph.
  auto range = [&](int ph, int& u0, int& u1) {
    const long U = a.U[ph];
    u0 = (int)(U * cta / G);
    u1 = (int)(U * (cta + 1) / G);
  };

  if (warp == 0) {
    // ---------------- weight producer: every tile of the solve, in order ----
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      long it = 0;
      bool ok = true;
      for (int k = 0; k < a.S && ok; ++k)
        for (int l = 0; l < L && ok; ++l)
          for (int ph = 0; ph < 4 && ok; ++ph) {
            int u0, u1;
            range(ph, u0, u1);
            const CUtensorMap* map = ph == 0 ? &tmW0 : ph == 1 ? &tmW1 : ph == 2 ? &tmW2 : &tmW3;
            const int nkb = a.nkb[ph];
            for (int u = u0; u < u1; ++u, ++it) {
              const int s = (int)(it % R);
              if (it >= R) {
                const uint32_t par = (uint32_t)((it / R) - 1) & 1u;
                const uint64_t t0 = globaltimer_ns();
                const uint64_t lim = wait_limit_ns(a.status);
                while (!mbar_try_wait(&empty[s], par)) {
                  if (*s_stop || globaltimer_ns() - t0 > lim) {
                    if (!*s_stop) latch_error(a.status, VLA_DEV_TIMEOUT);
                    ok = false;
                    break;
                  }
                }
                if (!ok) break;
              }
              mbar_arrive_expect_tx(&full[s], kStage);
              tma_load_2d_hint(ring + (size_t)s * kStage, map, &full[s], (u % nkb) * 64,
                               l * a.N[ph] + (u / nkb) * 128, pol);
            }
          }
      // Nothing may land in shared memory after the CTA exits: wait for the
      // copies still in flight (the last R issued).
      const long first = it > R ? it - R : 0;
      for (long i = first; i < it; ++i) mbar_drain(&full[i % R], (uint32_t)(i / R) & 1u);
    }
  } else {
    // ---------------- warps 1..7: phases ------------------------------------
    const int wt = threadIdx.x - 32;  // 0..223
    unsigned bar_target = 0;
    int mma_phase = 0, att_phase = 0;
    long it = 0;  // ring stages consumed (MMA thread; -1 once a wait gave up)
    // completions so far of the two (Q, K) buffers' barriers kbar / qkfree
    // (the same count for both), of mma_done and of the per-unit attention
    // barriers: every work thread keeps them (phase parities), thread 32 also
    // drains them before the CTA exits
    int xbase[2] = {0, 0}, n_mma = 0, n_att = 0;
    bool ok = true;
    auto barrier = [&]() {
      bar_target += (unsigned)G;
      if (ok) ok = grid_sync(a, bar_target, s_fail);
      else {  // keep the arrival count consistent for the CTAs still running
        tc_fence_before();
        named_bar_sync(kBarWork, kWork);
        if (threadIdx.x == 64) atomicAdd(a.bar, 1u);
        named_bar_sync(kBarWork, kWork);
      }
    };

    // ---- token rms of the residual stream: CTA t < T owns token t -------
    auto token_rms = [&](float* dst) {
      if (cta < T) {
        const float* hr = a.h + (size_t)cta * D;
        float ss = 0.f;
        for (int i = wt * 4; i < D; i += kWork * 4) {
          const float4 v = ldcg4(hr + i);
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = work_sum(ss, red);
        if (wt == 0) __stcg(dst + cta, rsqrtf(ss / (float)D + a.eps));
      }
    };
    // ---- zero an fp32 buffer of n floats, split over the grid -------------
    auto zero_buf = [&](float* p, long n) {
      const long per = ((n / 4 + G - 1) / G) * 4;
      const long b0 = per * cta, b1 = b0 + per < n ? b0 + per : n;
      for (long i = b0 + wt * 4; i < b1; i += kWork * 4) stcg4(p + i, make_float4(0.f, 0.f, 0.f, 0.f));
    };
    // ---- h[t] = x[t] W_in^T for token t = cta ------------------------------
    auto embed_token = [&](const float* x) {
      if (cta < T) {
        for (int j = wt; j < a.d_a; j += kWork) xs[j] = x[(size_t)cta * a.d_a + j];
        named_bar_sync(kBarWork, kWork);
        for (int i = wt; i < D; i += kWork) {
          const float* w = a.win + (size_t)i * a.d_a;
          float acc = 0.f;
          for (int j = 0; j < a.d_a; ++j) acc += xs[j] * __ldg(w + j);
          __stcg(a.h + (size_t)cta * D + i, acc);
        }
        named_bar_sync(kBarWork, kWork);
      }
    };

    // ---- one linear phase ----------------------------------------------------
    // ph 0: [W_q;W_k;W_v] (B = (1 + gamma_a) h) -> acc_qkv
    // ph 1: W_o (B = merged attention output)   -> h
    // ph 2: W_up (B = (1 + gamma_m) h)          -> acc_up
    // ph 3: W_down (B = GeLU(r_m acc_up + W_up beta_m)) -> h
    auto linear = [&](int ph, int k, int l) {
      int u0, u1;
      range(ph, u0, u1);
      const int len = u1 - u0;
      if (len <= 0) return;
      const int nkb = a.nkb[ph], N = a.N[ph];
      const int kb0 = u0 % nkb;
      const int ntiles = len < nkb ? len : nkb;
      const uint32_t btile = (uint32_t)BN * 128u;
      const float* gam = a.modtab + ((size_t)(k * L + l) * 4 + (ph == 0 ? 0 : 2)) * D;
      const float* cup = a.cup + (size_t)(k * L + l) * a.F;
      // 1. B operand tiles (one per distinct K block of the range)
      const int nchunks = ntiles * BN * 8;
      for (int idx = wt; idx < nchunks; idx += kWork) {
        const int s = idx / (BN * 8), rem = idx - s * BN * 8, row = rem >> 3, c = rem & 7;
        const int kb = (kb0 + s) % nkb, col = kb * 64 + c * 8;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
        if (row < T) {
          if (ph == 0 || ph == 2) {
            const float* hp = a.h + (size_t)row * D + col;
            const float4 h0 = ldcg4(hp), h1 = ldcg4(hp + 4);
            const float4 g0 = __ldg((const float4*)(gam + col)), g1 = __ldg((const float4*)(gam + col + 4));
            v[0] = h0.x * (1.f + g0.x); v[1] = h0.y * (1.f + g0.y); v[2] = h0.z * (1.f + g0.z);
            v[3] = h0.w * (1.f + g0.w); v[4] = h1.x * (1.f + g1.x); v[5] = h1.y * (1.f + g1.y);
            v[6] = h1.z * (1.f + g1.z); v[7] = h1.w * (1.f + g1.w);
          } else if (ph == 3) {
            const float r = __ldcg(a.rms + a.T + row);
            const float* ap = a.accu + (size_t)row * a.F + col;
            const float4 x0 = ldcg4(ap), x1 = ldcg4(ap + 4);
            const float4 c0 = __ldg((const float4*)(cup + col)), c1 = __ldg((const float4*)(cup + col + 4));
            v[0] = gelu_exact(fmaf(r, x0.x, c0.x)); v[1] = gelu_exact(fmaf(r, x0.y, c0.y));
            v[2] = gelu_exact(fmaf(r, x0.z, c0.z)); v[3] = gelu_exact(fmaf(r, x0.w, c0.w));
            v[4] = gelu_exact(fmaf(r, x1.x, c1.x)); v[5] = gelu_exact(fmaf(r, x1.y, c1.y));
            v[6] = gelu_exact(fmaf(r, x1.z, c1.z)); v[7] = gelu_exact(fmaf(r, x1.w, c1.w));
          } else {
            // merge the attention chunks of this (token, head) row
            const int j = col / a.d_h, dcol = col - j * a.d_h;
            const int g = j / a.group, jj = j - g * a.group;
            const int b = row / a.H, i = row - b * a.H;
            const int r = jj * a.H + i, qt = r >> 7, lr = r & 127;
            const long ub = ((long)(b * a.n_kv + g) * a.nqt + qt) * a.nch;
            float M = -INFINITY;
            for (int ch = 0; ch < a.nch; ++ch) M = fmaxf(M, __ldcg(&a.oml[(ub + ch) * 128 + lr].x));
            float den = 0.f;
            for (int ch = 0; ch < a.nch; ++ch) {
              const float2 ml = __ldcg(&a.oml[(ub + ch) * 128 + lr]);
              const float wgt = fast_exp2(ml.x - M);
              den += wgt * ml.y;
              float o[8];
              unpack8(__ldcg((const uint4*)(a.opart + ((ub + ch) * 128 + lr) * a.d_h + dcol)), o);
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] += wgt * o[e];
            }
            const float inv = 1.f / den;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] *= inv;
          }
        }
        st_shared_v4_u32(smem_u32(work + (size_t)s * btile) + sw128_offset((uint32_t)row, (uint32_t)c), pack8(v));
      }
      fence_proxy_async_smem();
      named_bar_sync(kBarWork, kWork);
      // 2. MMAs (one thread): D[seg] (+)= W tile x B tile
      if (threadIdx.x == 32) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, BN);
        for (int u = u0; u < u1 && it >= 0; ++u, ++it) {
          const int seg = u / nkb - u0 / nkb, kb = u % nkb;
          const int slot = (kb - kb0 + nkb) % nkb;
          const int s = (int)(it % R);
          if (!mbar_wait(&full[s], (uint32_t)(it / R) & 1u, a.status)) {
            *s_fail = 1;  // the phase's result is lost; the grid barrier reports it
            it = -1;      // stop consuming: later stages would be out of order
            break;
          }
          tc_fence_after();
          const bool first = (u == u0) || (kb == 0);
          const uint32_t aa = smem_u32(ring + (size_t)s * kStage), bb = smem_u32(work + (size_t)slot * btile);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            umma_bf16(tmem + (uint32_t)(seg * BN), sdesc_k128(aa + k4 * 32), sdesc_k128(bb + k4 * 32), idesc,
                      (!first || k4 > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        umma_commit(mma_done);
        ++n_mma;
      }
      // 3. epilogue: add the partial sums into the fp32 output
      if (warp >= 4) {
        const bool w_ok = __all_sync(0xffffffffu, mbar_wait(mma_done, (uint32_t)mma_phase & 1u, a.status) && !*s_fail);
        tc_fence_after();
        if (w_ok) {
          float* out = ph == 0 ? a.accq : (ph == 2 ? a.accu : a.h);
          const int row = (warp - 4) * 32 + lane;
          const int nseg = (u1 - 1) / nkb - u0 / nkb + 1;
          for (int seg = 0; seg < nseg; ++seg) {
            const int n = (u0 / nkb + seg) * 128 + row;
            const uint32_t taddr = tmem + ((uint32_t)((warp - 4) * 32) << 16) + (uint32_t)(seg * BN);
            for (int c0 = 0; c0 < T; c0 += 16) {
              float v[16];
              tmem_ld16(taddr + (uint32_t)c0, v);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < T) red_add_f32(out + (size_t)(c0 + j) * N + n, v[j]);
            }
          }
        } else {
          *s_fail = 1;
        }
      }
      ++mma_phase;
    };

    // ---- one attention unit ----------------------------------------------------
    auto attention = [&](int unit, int k, int l) {
      const int ch = unit % a.nch;
      int rest = unit / a.nch;
      const int qt = rest % a.nqt;
      rest /= a.nqt;
      const int g = rest % a.n_kv, b = rest / a.n_kv;
      const int rows = a.group * a.H - qt * 128 < 128 ? a.group * a.H - qt * 128 : 128;
      const int k0 = ch * kKC;
      const int nkeys = a.P + a.H - k0 < kKC ? a.P + a.H - k0 : kKC;
      int npre = a.P - k0;
      npre = npre < 0 ? 0 : (npre > nkeys ? nkeys : npre);
      const int z = (l * a.B + b) * a.n_kv + g;
      const int dh = a.d_h, nsub = dh / 64;
      const float* cq = a.cqkv + (size_t)(k * L + l) * a.qkvdim;
      const float* rms_a = a.rms;
      const uint32_t tS = tmem + 256u, tO = tmem;
      const uint64_t pol_kv = l2_policy_evict_last();
      // S = Q K^T over d_h / 64 sub-tiles, two buffers of (Q_s, K_s)
      for (int s = 0; s < nsub; ++s) {
        const int buf = s & 1;
        uint8_t* Qs = work + (size_t)buf * 32768;
        uint8_t* Ks = Qs + 16384;
        // the MMAs of sub-tile s - 2 have read this buffer
        if (s >= 2 && !mbar_wait(&qkfree[buf], (uint32_t)(xbase[buf] + ((s - 2) >> 1)) & 1u, a.status)) *s_fail = 1;
        if (threadIdx.x == 32) {
          mbar_arrive_expect_tx(&kbar[buf], (uint32_t)kKC * 128u);
          tma_load_3d_hint(Ks, &tmK, &kbar[buf], s * 64, k0, z, pol_kv);
        }
        for (int idx = wt; idx < 128 * 8; idx += kWork) {
          const int r = idx >> 3, c = idx & 7;
          float v[8];
          if (r < rows) {
            const int qr = qt * 128 + r, jj = qr / a.H, i = qr - jj * a.H, t = b * a.H + i;
            const int n = (g * a.group + jj) * dh + s * 64 + c * 8;
            const float rr = __ldcg(rms_a + t);
            const float4 x0 = ldcg4(a.accq + (size_t)t * a.qkvdim + n), x1 = ldcg4(a.accq + (size_t)t * a.qkvdim + n + 4);
            const float4 c0 = __ldg((const float4*)(cq + n)), c1 = __ldg((const float4*)(cq + n + 4));
            v[0] = fmaf(rr, x0.x, c0.x); v[1] = fmaf(rr, x0.y, c0.y); v[2] = fmaf(rr, x0.z, c0.z);
            v[3] = fmaf(rr, x0.w, c0.w); v[4] = fmaf(rr, x1.x, c1.x); v[5] = fmaf(rr, x1.y, c1.y);
            v[6] = fmaf(rr, x1.z, c1.z); v[7] = fmaf(rr, x1.w, c1.w);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
          }
          st_shared_v4_u32(smem_u32(Qs) + sw128_offset((uint32_t)r, (uint32_t)c), pack8(v));
        }
        // action-token keys of this chunk (rows npre..nkeys-1), after the TMA
        // of the cached rows has landed (it zero-fills rows past the prefix)
        if (!mbar_wait(&kbar[buf], (uint32_t)(xbase[buf] + (s >> 1)) & 1u, a.status)) *s_fail = 1;
        for (int idx = wt; idx < (nkeys - npre) * 8; idx += kWork) {
          const int jr = npre + (idx >> 3), c = idx & 7;
          const int t = b * a.H + (k0 + jr - a.P);
          const int n = a.qdim + g * dh + s * 64 + c * 8;
          const float rr = __ldcg(rms_a + t);
          const float4 x0 = ldcg4(a.accq + (size_t)t * a.qkvdim + n), x1 = ldcg4(a.accq + (size_t)t * a.qkvdim + n + 4);
          const float4 c0 = __ldg((const float4*)(cq + n)), c1 = __ldg((const float4*)(cq + n + 4));
          float v[8] = {fmaf(rr, x0.x, c0.x), fmaf(rr, x0.y, c0.y), fmaf(rr, x0.z, c0.z), fmaf(rr, x0.w, c0.w),
                        fmaf(rr, x1.x, c1.x), fmaf(rr, x1.y, c1.y), fmaf(rr, x1.z, c1.z), fmaf(rr, x1.w, c1.w)};
          st_shared_v4_u32(smem_u32(Ks) + sw128_offset((uint32_t)jr, (uint32_t)c), pack8(v));
        }
        fence_proxy_async_smem();
        named_bar_sync(kBarWork, kWork);
        if (threadIdx.x == 32) {
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(128, kKC);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            umma_bf16(tS, sdesc_k128(smem_u32(Qs) + k4 * 32), sdesc_k128(smem_u32(Ks) + k4 * 32), idesc,
                      (s > 0 || k4 > 0) ? 1u : 0u);
          umma_commit(&qkfree[buf]);
          if (s == nsub - 1) umma_commit(sdone);
        }
      }
      // V^T of the chunk into the (now free) Q/K buffers: 2 x [d_h][64 keys]
      uint8_t* Vt = work;
      uint8_t* Ps = work + 65536;
      const uint32_t att_par = (uint32_t)att_phase & 1u;
      if (threadIdx.x == 32) {
        if (!mbar_wait(sdone, att_par, a.status)) *s_fail = 1;
        mbar_arrive_expect_tx(vbar, 2u * (uint32_t)dh * 128u);
        for (int kh = 0; kh < 2; ++kh)
          tma_load_3d_hint(Vt + (size_t)kh * dh * 128, &tmVt, vbar, k0 + kh * 64, 0, z, pol_kv);
      }
      if (warp >= 4) {
        // softmax of this unit's rows: one row per thread
        const int row = (warp - 4) * 32 + lane;
        if (!mbar_wait(sdone, att_par, a.status)) *s_fail = 1;
        tc_fence_after();
        const uint32_t taddr = tS + ((uint32_t)((warp - 4) * 32) << 16);
        float sv[kKC];
#pragma unroll
        for (int q = 0; q < kKC / 16; ++q) tmem_ld16(taddr + (uint32_t)(q * 16), sv + q * 16);
        const bool live = row < rows;
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < kKC; ++j)
          if (j < nkeys) m = fmaxf(m, sv[j] * a.scale_log2);
        if (!live) m = 0.f;
        float lsum = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < kKC / 8; ++c8) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = c8 * 8 + e;
            p[e] = (live && j < nkeys) ? fast_exp2(sv[j] * a.scale_log2 - m) : 0.f;
          }
          const uint4 pk = pack8(p);
          // the sum uses the bf16 values the P V product multiplies
          float pb[8];
          unpack8(pk, pb);
#pragma unroll
          for (int e = 0; e < 8; ++e) lsum += pb[e];
          st_shared_v4_u32(smem_u32(Ps + (size_t)(c8 >> 3) * 16384) + sw128_offset((uint32_t)row, (uint32_t)(c8 & 7)),
                           pk);
        }
        rowml[row] = make_float2(m, lsum);
        fence_proxy_async_smem();
        tc_fence_before();
      } else {
        // warps 1..3: the action tokens' values into V^T once the cached rows landed
        if (!mbar_wait(vbar, att_par, a.status)) *s_fail = 1;
        const int bt = threadIdx.x - 32;  // 0..95
        for (int idx = bt; idx < (nkeys - npre) * (dh / 8); idx += 96) {
          const int jr = npre + idx / (dh / 8), d8 = (idx % (dh / 8)) * 8;
          const int t = b * a.H + (k0 + jr - a.P);
          const int n = a.qdim + a.kvdim + g * dh + d8;
          const float rr = __ldcg(rms_a + t);
          const float4 x0 = ldcg4(a.accq + (size_t)t * a.qkvdim + n), x1 = ldcg4(a.accq + (size_t)t * a.qkvdim + n + 4);
          const float4 c0 = __ldg((const float4*)(cq + n)), c1 = __ldg((const float4*)(cq + n + 4));
          const float v[8] = {fmaf(rr, x0.x, c0.x), fmaf(rr, x0.y, c0.y), fmaf(rr, x0.z, c0.z), fmaf(rr, x0.w, c0.w),
                              fmaf(rr, x1.x, c1.x), fmaf(rr, x1.y, c1.y), fmaf(rr, x1.z, c1.z), fmaf(rr, x1.w, c1.w)};
          uint8_t* half = Vt + (size_t)(jr >> 6) * dh * 128;
          const int kk = jr & 63;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t off = sw128_offset((uint32_t)(d8 + e), (uint32_t)(kk >> 3)) + (uint32_t)(kk & 7) * 2u;
            *(bf16*)(half + off) = __float2bfloat16_rn(v[e]);
          }
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(kBarWork, kWork);
      // O = P V
      if (threadIdx.x == 32) {
        if (!mbar_wait(vbar, att_par, a.status)) *s_fail = 1;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, dh);
        for (int kk = 0; kk < kKC / 16; ++kk) {
          const uint32_t pa = smem_u32(Ps + (size_t)(kk >> 2) * 16384) + (uint32_t)(kk & 3) * 32u;
          const uint32_t va = smem_u32(Vt + (size_t)(kk >> 2) * dh * 128) + (uint32_t)(kk & 3) * 32u;
          umma_bf16(tO, sdesc_k128(pa), sdesc_k128(va), idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(odone);
        ++n_att;
      }
      if (warp >= 4) {
        const int row = (warp - 4) * 32 + lane;
        if (!mbar_wait(odone, att_par, a.status)) *s_fail = 1;
        tc_fence_after();
        const uint32_t taddr = tO + ((uint32_t)((warp - 4) * 32) << 16);
        bf16* dst = a.opart + ((size_t)unit * 128 + row) * dh;
        for (int c0 = 0; c0 < dh; c0 += 16) {
          float v[16];
          tmem_ld16(taddr + (uint32_t)c0, v);
          if (row < rows) {
            __stcg((uint4*)(dst + c0), pack8(v));
            __stcg((uint4*)(dst + c0 + 8), pack8(v + 8));
          }
        }
        if (row < rows) __stcg(&a.oml[(size_t)unit * 128 + row], rowml[row]);
        tc_fence_before();
      }
      // the next unit reuses the buffers that P V read: wait for the epilogue
      named_bar_sync(kBarWork, kWork);
      xbase[0] += (nsub + 1) >> 1;
      xbase[1] += nsub >> 1;
      ++att_phase;
    };

    // ---- head: final norm, W_out, Euler update, next chunk's W_in ---------
    auto head = [&](int k) {
      if (cta < T) {
        const int t = cta;
        const float* hr = a.h + (size_t)t * D;
        float ss = 0.f;
        for (int i = wt; i < D; i += kWork) {
          const float hv = __ldcg(hr + i);
          hrow[i] = hv;
          ss += hv * hv;
        }
        ss = work_sum(ss, red);
        const float r = rsqrtf(ss / (float)D + a.eps);
        const float* gf = a.modf + (size_t)k * 2 * D;
        const float* bf = gf + D;
        for (int i = wt; i < D; i += kWork) hrow[i] = hrow[i] * r * (1.f + __ldg(gf + i)) + __ldg(bf + i);
        named_bar_sync(kBarWork, kWork);
        const float dt = (float)((double)(k + 1) / a.S - (double)k / a.S);
        const float* x_in = k == 0 ? a.noise : a.actions;
        for (int o = warp - 1; o < a.d_a; o += 7) {
          const float* w = a.wout + (size_t)o * D;
          float acc = 0.f;
          for (int i = lane; i < D; i += 32) acc += hrow[i] * __ldg(w + i);
          acc = warp_sum(acc);
          if (lane == 0) {
            const size_t idx = (size_t)t * a.d_a + o;
            const float xn = fmaf(dt, acc, x_in[idx]);
            a.actions[idx] = xn;
            if (a.vtap) a.vtap[(size_t)k * T * a.d_a + idx] = acc;
            xs[o] = xn;
          }
        }
        named_bar_sync(kBarWork, kWork);
        if (k + 1 < a.S) {
          for (int i = wt; i < D; i += kWork) {
            const float* w = a.win + (size_t)i * a.d_a;
            float acc = 0.f;
            for (int j = 0; j < a.d_a; ++j) acc += xs[j] * __ldg(w + j);
            __stcg(a.h + (size_t)t * D + i, acc);
          }
        }
      }
      if (cta == 0 && wt == 0 && a.abort && *a.abort) {
        latch_error(a.status, VLA_DEV_ABORTED);
        __stcg(a.stop, 1);
      }
    };

    // ---- the solve ------------------------------------------------------------
    embed_token(a.noise);
    zero_buf(a.accq, (long)T * a.qkvdim);
    zero_buf(a.accu, (long)T * a.F);
    barrier();
    for (int k = 0; k < a.S && ok; ++k) {
      for (int l = 0; l < L && ok; ++l) {
        linear(0, k, l);                      // A
        token_rms(a.rms);
        zero_buf(a.accu, (long)T * a.F);
        barrier();
        for (int u = cta; u < a.att_units && ok; u += G) attention(u, k, l);  // B
        barrier();
        linear(1, k, l);                      // C
        zero_buf(a.accq, (long)T * a.qkvdim);
        barrier();
        linear(2, k, l);                      // D
        token_rms(a.rms + T);
        barrier();
        linear(3, k, l);                      // E
        barrier();
      }
      if (!ok) break;
      head(k);
      barrier();
      if (ok && __ldcg(a.stop)) break;  // abort seen at this step boundary (uniform)
    }
    if (threadIdx.x == 32) {
      *s_stop = 1;
      // Before TMEM is freed and the CTA exits, every MMA and copy this thread
      // issued must be complete (they are, unless a wait gave up): wait for
      // the last completion of each barrier.
      if (n_mma) mbar_drain(mma_done, (uint32_t)(n_mma - 1) & 1u);
      for (int i = 0; i < 2; ++i)
        if (xbase[i]) {
          mbar_drain(&kbar[i], (uint32_t)(xbase[i] - 1) & 1u);
          mbar_drain(&qkfree[i], (uint32_t)(xbase[i] - 1) & 1u);
        }
      if (n_att) {
        mbar_drain(sdone, (uint32_t)(n_att - 1) & 1u);
        mbar_drain(vbar, (uint32_t)(n_att - 1) & 1u);
        mbar_drain(odone, (uint32_t)(n_att - 1) & 1u);
      }
    }
  }
  // ---- teardown ----------------------------------------------------------------
  __syncthreads();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t persist_smem_bytes(int D) { return 1024 + persist_layout(D).total; }
int persist_ring_stages(int D) { return persist_layout(D).R; }

cudaError_t persist_init() { return set_max_dyn_smem(k_solver_persist); }

// CTAs of the kernel that fit on one SM with its shared memory (a
// cooperative launch of one CTA per SM needs 1).
cudaError_t persist_blocks_per_sm(int D, int* n) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k_solver_persist, kThreads, persist_smem_bytes(D));
}

cudaError_t launch_persist(const CUtensorMap* tmW, const CUtensorMap* tmK, const CUtensorMap* tmVt,
                           const PersistArgs& a, int grid, cudaStream_t st) {
  const size_t smem = persist_smem_bytes(a.D);
  if (smem > 227 * 1024 || persist_ring_stages(a.D) < 4) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(a.bar, 0, 2 * sizeof(unsigned), st);  // barrier counter and stop word
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_solver_persist, tmW[0], tmW[1], tmW[2], tmW[3], *tmK, *tmVt, a);
}
