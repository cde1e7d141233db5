// The whole S-step Euler solve of a few-token request as ONE persistent
// kernel ("vla.cpp: A Unified Inference Runtime for Vision-Language-Action
// Models", §III-A Eq. (1) integrated over the cached prefix of §III-B Eq. (2);
// the solver loop as a single launch of the latency model, Eq. (3)).
//
// At batch 1 the velocity network is bound by its weight bytes: every Euler
// step streams each token-dependent weight once and does little arithmetic
// with it.  A chain of one kernel per linear map pays a launch boundary, a
// first-load latency and a split-K exchange per map, several times the time
// the map's weights take over HBM.  Here one CTA per SM lives for the whole
// solve (cooperative launch, so every CTA is resident).  The work of a layer
// runs in phases separated by grid-wide barriers:
//   A   [W_q;W_k;W_v] over the modulated-norm input          -> acc_qkv (fp32)
//   B1  q, k_s, v_s^T = r acc_qkv + W beta (bf16), every CTA  -> workspace
//   B2  joint attention per (query tile, 128-key chunk)      -> partial O, (m, l)
//   B3  merge of the chunks, every CTA                        -> o (bf16)
//   C   W_o over o                                            -> h += (residual)
//   D   W_up over the modulated-norm input                    -> acc_up (fp32)
//   E   W_down over GeLU(r acc_up + W_up beta)                -> h += (residual)
// and one head phase per step (final norm, W_out, Euler update, and the input
// projection of the next step's chunk).
//
// CTA roles.  The last NA CTAs run the attention units (B2) and the token
// statistics; they hold no weight ring, so their whole shared memory takes a
// unit's Q, K and V^T tiles at once.  The other CTAs run the linear phases.
//
// Weight streaming.  Weights do not depend on activations, so on every linear
// CTA warp 0 streams each weight tile the CTA will multiply, in consumption
// order, into a ring of 128 x 64 bf16 stages, independently of the phases:
// while the CTA waits at a barrier or the attention runs, its next phases'
// weights are already arriving.  The work of each linear phase is the list of
// (128-row tile, 64-wide K block) units of its weight matrix, cut into equal
// contiguous ranges for the linear CTAs, so every SM streams the same number
// of weight bytes.  A CTA's partial sums are added into the fp32 output by
// bulk tensor reductions (one TMA reduce-add of a [tokens][128 rows] tile per
// segment, performed in L2), which also performs the residual additions of C
// and E.  (The order of those additions varies from run to run, so results
// agree to fp32 rounding, not bit for bit.)  Operand tiles are brought in by
// TMA as well (the fp32 rows of h or acc_up, converted in shared memory; o
// directly in the MMA's bf16 layout).
//
// The modulated RMSNorm is factored out of the GEMM: with
// u = h r (1 + gamma) + beta,  y = W u = r (W ((1 + gamma) h)) + W beta,
// so the B operand is bf16((1 + gamma) h) (no row statistics needed before
// the product), the row scale r = 1 / rms(h) is applied by the consumer of
// the sums, and W beta is a per-(step, layer) vector computed once per handle.
// The attention CTAs compute r during the phases that multiply (A, D).
//
// Attention unit: S = Q K^T on tcgen05 (Q, K by TMA from the bf16 workspace
// and the cache), softmax in fp32 (one row per thread), P in bf16, O = P V on
// tcgen05; the unit writes its unnormalised O (fp32) with the row maximum m
// and sum l, and B3 forms o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
//
// Warp roles (256 threads): warp 0 lane 0 streams weights; warp 1 lane 0
// issues MMAs and operand TMAs; warp 2 lane 0 runs the grid barrier; warps
// 1-7 build operands; warps 4-7 run epilogues and the softmax (TMEM lane
// quarter = warp % 4).
#include <math.h>

#include "vla_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWork = 224;             // threads of warps 1..7
constexpr uint32_t kStage = 16384;     // one 128 x 64 bf16 weight tile
constexpr int kKC = 128;               // keys per attention unit
constexpr uint32_t kHdr = 1024;        // header: TMEM slot, flags, reduction slots, x
constexpr uint32_t kSmemUse = 227u * 1024u - 1024u;  // usable dynamic shared memory (after alignment)
constexpr int kBarWork = 1;            // named barrier over warps 1..7
constexpr int kBarEpi = 2;             // named barrier over warps 4..7

// Linear CTAs: [header][work: B tiles + fp32 staging][mbarriers][head row:
// D floats][ring].
struct PLayout {
  uint32_t work, bars, hrow, ring;
  int R;
};
__host__ __device__ inline PLayout persist_layout(int D, uint32_t work_bytes) {
  PLayout s;
  s.work = kHdr;
  s.bars = s.work + ((work_bytes + 1023u) & ~1023u);
  s.hrow = s.bars + 64 * 8;
  s.ring = (s.hrow + (uint32_t)D * 4u + 1023u) & ~1023u;
  int R = s.ring < kSmemUse ? (int)((kSmemUse - s.ring) / kStage) : 0;
  s.R = R > 16 ? 16 : R;
  return s;
}
// Attention CTAs: [header][Q][K][V^T][P][mbarriers].
struct ALayout {
  uint32_t q, k, v, p, bars, end;
};
__host__ __device__ inline ALayout att_layout(int dh) {
  ALayout s;
  s.q = kHdr;
  s.k = s.q + 128u * (uint32_t)dh * 2u;
  s.v = s.k + (uint32_t)kKC * (uint32_t)dh * 2u;
  s.p = s.v + (uint32_t)dh * (uint32_t)kKC * 2u;
  s.bars = s.p + 128u * (uint32_t)kKC * 2u;
  s.end = s.bars + 8 * 8;
  return s;
}

// ---------------------------------------------------------------------------
// Small PTX helpers local to this kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const void* map, uint64_t* bar, int x, int y, int z,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// Bulk tensor reduction: add the shared-memory tile (box of the map) into the
// fp32 tensor at {x, y}; the addition is performed in L2.
__device__ __forceinline__ void tma_reduce_add_2d(const void* map, uint32_t ssrc, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   (uint64_t)map),
               "r"(x), "r"(y), "r"(ssrc)
               : "memory");
}
// Wait until this thread's bulk operations have completed and order their
// global writes (async proxy) before its later generic-proxy operations.
__device__ __forceinline__ void bulk_wait_all_writes() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Order this thread's earlier generic-proxy accesses (the barrier's acquire)
// before its later async-proxy (TMA) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
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
    uint64_t lim = 0;  // the handle's limit, read only once the wait has lasted 100 us
    for (uint32_t it = 1;; ++it) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.bar) : "memory");
      if (v >= target) break;
      if ((it & 63u) == 0) {
        const uint64_t el = globaltimer_ns() - t0;
        if (el > 100000ull) {
          if (!lim) lim = wait_limit_ns(a.status);
          if (el > lim) {
            latch_error(a.status, VLA_DEV_TIMEOUT);
            *fail = 1;
            break;
          }
          if (*(volatile int*)a.status == VLA_DEV_TIMEOUT) {
            *fail = 1;
            break;
          }
        }
      }
    }
    __threadfence();
  }
  named_bar_sync(kBarWork, kWork);
  tc_fence_after();
  return *fail == 0;
}

// Optional phase trace (built only with -DVLA_PERSIST_TRACE): thread `thr`
// of every CTA stamps %globaltimer at event `ev` (< 8) of phase `ph` of
// solver step 1 into trace[(cta * 160 + ph) * 8 + ev].
#ifdef VLA_PERSIST_TRACE
#define PTRACE_T(thr, k, ph, ev)                                                     \
  do {                                                                             \
    if (a.trace && (k) == 1 && threadIdx.x == (thr) && (ph) < 160)                   \
      a.trace[((size_t)blockIdx.x * 160 + (ph)) * 8 + (ev)] = globaltimer_ns();     \
  } while (0)
#else
#define PTRACE_T(thr, k, ph, ev) \
  do {                           \
  } while (0)
#endif
#define PTRACE(k, ph, ev) PTRACE_T(64, k, ph, ev)

struct Maps {
  CUtensorMap w[4];  // bf16 weights, box 64 x 128 (SW128)
  CUtensorMap kc;    // K_C {d_h, P, L*B*n_kv}, box 64 x 128 (SW128)
  CUtensorMap vc;    // V_C^T {P, d_h, L*B*n_kv}, box 64 x d_h (SW128)
  CUtensorMap ks;    // k_s {d_h, H, B*n_kv}, box 64 x 128 (SW128)
  CUtensorMap vs;    // v_s^T {H, d_h, B*n_kv}, box 64 x d_h (SW128)
  CUtensorMap q;     // q [B*n_q*H][d_h], box 64 x 128 (SW128)
  CUtensorMap hld;   // h [T][D] fp32, box 64 x BN (operand loads)
  CUtensorMap uld;   // acc_up [T][F] fp32, box 64 x BN
  CUtensorMap old;   // o [T][qdim] bf16, box 64 x BN (SW128)
  CUtensorMap red[3];  // acc_qkv, h, acc_up fp32, box 128 x BN (reductions)
};

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) k_solver_persist(const __grid_constant__ Maps m, const PersistArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int NA = a.n_att, GL = G - NA;
  const bool att_cta = cta >= GL;
  const int T = a.T, D = a.D, L = a.L, BN = a.BN;
  // header
  uint32_t* tmem_slot = (uint32_t*)smem;
  volatile int* s_fail = (volatile int*)(smem + 16);  // a wait gave up: leave
  volatile int* s_stop = (volatile int*)(smem + 20);  // tells the weight producer to stop
  float* red = (float*)(smem + 32);                   // [8]
  float* xs = (float*)(smem + 64);                    // [64] next chunk of one token
  // linear CTAs
  const PLayout Ls = persist_layout(D, (uint32_t)a.work_bytes);
  const int R = Ls.R;
  uint8_t* work = smem + Ls.work;
  uint8_t* ring = smem + Ls.ring;
  float* hrow = (float*)(smem + Ls.hrow);
  float* rsum = (float*)work;    // [7][64] head reductions (the work region is idle then)
  uint64_t* lb = (uint64_t*)(smem + Ls.bars);
  uint64_t* full = lb;           // [16]
  uint64_t* empty = lb + 16;     // [16]
  uint64_t* mma_done = lb + 32;
  uint64_t* bbar = lb + 33;      // operand tiles landed
  // attention CTAs
  const ALayout As = att_layout(a.d_h);
  uint64_t* ab = (uint64_t*)(smem + As.bars);
  uint64_t* qkbar = ab;          // Q and K tiles landed
  uint64_t* vbar = ab + 1;       // V^T tile landed
  uint64_t* sdone = ab + 2;
  uint64_t* odone = ab + 3;

  if (threadIdx.x == 0) {
    if (!att_cta) {
      for (int i = 0; i < R; ++i) {
        mbar_init(&full[i], 1);
        mbar_init(&empty[i], 1);
      }
      mbar_init(mma_done, 1);
      mbar_init(bbar, 1);
    } else {
      for (int i = 0; i < 4; ++i) mbar_init(&ab[i], 1);
    }
    *s_fail = 0;
    *s_stop = 0;
    fence_mbar_init();
    if (!att_cta) {
      for (int i = 0; i < 4; ++i) tma_prefetch_desc(&m.w[i]);
    } else {
      tma_prefetch_desc(&m.kc);
      tma_prefetch_desc(&m.vc);
      tma_prefetch_desc(&m.ks);
      tma_prefetch_desc(&m.vs);
      tma_prefetch_desc(&m.q);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Unit range of linear CTA `cta` in linear phase ph.
  auto range = [&](int ph, int& u0, int& u1) {
    const long U = a.U[ph];
    u0 = (int)(U * cta / GL);
    u1 = (int)(U * (cta + 1) / GL);
  };

  if (warp == 0) {
    // ---------------- weight producer: every tile of the solve, in order ----
    if (lane == 0 && !att_cta) {
      const uint64_t pol = l2_policy_evict_first();
      long it = 0;
      bool ok = true;
      for (int k = 0; k < a.S && ok; ++k)
        for (int l = 0; l < L && ok; ++l)
          for (int ph = 0; ph < 4 && ok; ++ph) {
            int u0, u1;
            range(ph, u0, u1);
            const int nkb = a.nkb[ph];
            for (int u = u0; u < u1; ++u, ++it) {
              const int s = (int)(it % R);
              if (it >= R) {
                const uint32_t par = (uint32_t)((it / R) - 1) & 1u;
                const uint64_t t0 = globaltimer_ns();
                uint64_t lim = 0;  // read once the wait has lasted 100 us
                while (!mbar_try_wait(&empty[s], par)) {
                  if (*s_stop) {
                    ok = false;
                    break;
                  }
                  const uint64_t el = globaltimer_ns() - t0;
                  if (el > 100000ull) {
                    if (!lim) lim = wait_limit_ns(a.status);
                    if (el > lim) {
                      latch_error(a.status, VLA_DEV_TIMEOUT);
                      ok = false;
                      break;
                    }
                  }
                }
                if (!ok) break;
              }
              mbar_arrive_expect_tx(&full[s], kStage);
              tma_load_2d_hint(ring + (size_t)s * kStage, &m.w[ph], &full[s], (u % nkb) * 64,
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
    int n_mma = 0, n_att = 0;  // commits issued by thread 32 (drained at exit)
    bool ok = true;
    int tk = -1, tph = 0;  // step and phase index within the step (trace)
    (void)tk;
    auto barrier = [&]() {
      PTRACE(tk, tph, 2);
      bar_target += (unsigned)G;
      if (ok) {
        ok = grid_sync(a, bar_target, s_fail);
      } else {  // keep the arrival count consistent for the CTAs still running
        tc_fence_before();
        named_bar_sync(kBarWork, kWork);
        if (threadIdx.x == 64) atomicAdd(a.bar, 1u);
        named_bar_sync(kBarWork, kWork);
      }
      PTRACE(tk, tph, 3);
      ++tph;
      PTRACE(tk, tph, 0);
    };

    // ---- token statistic r = 1 / rms(h) (attention CTAs) -------------------
    auto token_rms = [&](float* dst) {
      if (!att_cta) return;
      for (int t = cta - GL; t < T; t += NA) {
        const float* hr = a.h + (size_t)t * D;
        float ss = 0.f;
        for (int i = wt * 4; i < D; i += kWork * 4) {
          const float4 v = ldcg4(hr + i);
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = work_sum(ss, red);
        if (wt == 0) __stcg(dst + t, rsqrtf(ss / (float)D + a.eps));
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

    // ---- one linear phase (linear CTAs) -------------------------------------
    // ph 0: [W_q;W_k;W_v] (B = (1 + gamma_a) h) -> acc_qkv
    // ph 1: W_o (B = o, bf16 by TMA)            -> h
    // ph 2: W_up (B = (1 + gamma_m) h)          -> acc_up
    // ph 3: W_down (B = GeLU(r_m acc_up + W_up beta_m)) -> h
    auto linear = [&](int ph, int k, int l) {
      if (att_cta) return;
      int u0, u1;
      range(ph, u0, u1);
      const int len = u1 - u0;
      if (len <= 0) return;
      const int nkb = a.nkb[ph];
      const int kb0 = u0 % nkb;
      const int ntiles = len < nkb ? len : nkb;
      const uint32_t btile = (uint32_t)BN * 128u;
      uint8_t* stage = work + (size_t)ntiles * btile;  // fp32 operand rows, then the reduction tiles
      const uint32_t lpar = (uint32_t)mma_phase & 1u;
      // 1. operand tiles by TMA: o straight into the B tiles; fp32 rows of h /
      //    acc_up into the staging area for conversion
      if (threadIdx.x == 32) {
        fence_proxy_async_global();
        if (ph == 1) {
          mbar_arrive_expect_tx(bbar, (uint32_t)ntiles * btile);
          for (int s = 0; s < ntiles; ++s) tma_load_2d(work + (size_t)s * btile, &m.old, bbar, ((kb0 + s) % nkb) * 64, 0);
        } else {
          mbar_arrive_expect_tx(bbar, (uint32_t)ntiles * (uint32_t)BN * 256u);
          for (int s = 0; s < ntiles; ++s)
            tma_load_2d(stage + (size_t)s * BN * 256, ph == 3 ? &m.uld : &m.hld, bbar, ((kb0 + s) % nkb) * 64, 0);
        }
      }
      if (ph != 1) {
        // per-column constants (1 + gamma, or W_up beta) and the token scales,
        // fetched into shared memory while the operand rows are in flight
        const float* colc = ph == 3 ? a.cup + (size_t)(k * L + l) * a.F
                                    : a.modtab + ((size_t)(k * L + l) * 4 + (ph == 0 ? 0 : 2)) * D;
        float* cs = hrow;            // [ntiles * 64] column constants
        float* rs = hrow + 5 * 64;   // [BN] token scales (phase E)
        for (int i = wt; i < ntiles * 64; i += kWork) {
          const float v = __ldg(colc + ((kb0 + i / 64) % nkb) * 64 + (i & 63));
          cs[i] = ph == 3 ? v : 1.f + v;
        }
        if (ph == 3)
          for (int i = wt; i < BN; i += kWork) rs[i] = i < T ? __ldcg(a.rms + a.T + i) : 0.f;
        named_bar_sync(kBarWork, kWork);
        if (!mbar_wait(bbar, lpar, a.status)) *s_fail = 1;
        const int nchunks = ntiles * BN * 8;
        for (int idx = wt; idx < nchunks; idx += kWork) {
          const int s = idx / (BN * 8), rem = idx - s * BN * 8, row = rem >> 3, c = rem & 7;
          const float* src = (const float*)(stage + (size_t)s * BN * 256 + (size_t)row * 256 + c * 32);
          const float* cc = cs + s * 64 + c * 8;
          const float4 x0 = *(const float4*)src, x1 = *(const float4*)(src + 4);
          const float4 c0 = *(const float4*)cc, c1 = *(const float4*)(cc + 4);
          float v[8];
          if (ph == 3) {
            const float r = rs[row];  // 0 for padding rows: GeLU(c) there, then zeroed
            v[0] = gelu_exact(fmaf(r, x0.x, c0.x)); v[1] = gelu_exact(fmaf(r, x0.y, c0.y));
            v[2] = gelu_exact(fmaf(r, x0.z, c0.z)); v[3] = gelu_exact(fmaf(r, x0.w, c0.w));
            v[4] = gelu_exact(fmaf(r, x1.x, c1.x)); v[5] = gelu_exact(fmaf(r, x1.y, c1.y));
            v[6] = gelu_exact(fmaf(r, x1.z, c1.z)); v[7] = gelu_exact(fmaf(r, x1.w, c1.w));
            if (row >= T) {
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = 0.f;
            }
          } else {
            v[0] = x0.x * c0.x; v[1] = x0.y * c0.y; v[2] = x0.z * c0.z; v[3] = x0.w * c0.w;
            v[4] = x1.x * c1.x; v[5] = x1.y * c1.y; v[6] = x1.z * c1.z; v[7] = x1.w * c1.w;
          }
          st_shared_v4_u32(smem_u32(work + (size_t)s * btile) + sw128_offset((uint32_t)row, (uint32_t)c),
                           pack8(v));
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(kBarWork, kWork);
      PTRACE(k, tph, 1);
      // 2. MMAs (one thread): D[seg] (+)= W tile x B tile
      if (threadIdx.x == 32) {
        if (ph == 1 && !mbar_wait(bbar, lpar, a.status)) *s_fail = 1;
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
      // 3. epilogue: stage each segment's partial sums [token][128 rows] in
      // shared memory and add them into the fp32 output with one bulk tensor
      // reduction per segment (performed in L2)
      if (warp >= 4) {
        const bool w_ok = __all_sync(0xffffffffu, mbar_wait(mma_done, lpar, a.status) && !*s_fail);
        tc_fence_after();
        PTRACE_T(128, k, tph, 4);
        const int nseg = (u1 - 1) / nkb - u0 / nkb + 1;
        if (w_ok) {
          const int row = (warp - 4) * 32 + lane;
          for (int seg = 0; seg < nseg; ++seg) {
            const uint32_t taddr = tmem + ((uint32_t)((warp - 4) * 32) << 16) + (uint32_t)(seg * BN);
            float* stg = (float*)(stage + (size_t)seg * BN * 512);
            for (int c0 = 0; c0 < T; c0 += 16) {
              float v[16];
              tmem_ld16(taddr + (uint32_t)c0, v);
#pragma unroll
              for (int j = 0; j < 16; ++j) stg[(c0 + j) * 128 + row] = v[j];
            }
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        named_bar_sync(kBarEpi, 128);
        if (threadIdx.x == 128 && w_ok) {
          const CUtensorMap* rmap = ph == 0 ? &m.red[0] : (ph == 2 ? &m.red[2] : &m.red[1]);
          for (int seg = 0; seg < nseg; ++seg)
            tma_reduce_add_2d(rmap, smem_u32(stage) + (uint32_t)(seg * BN * 512), (u0 / nkb + seg) * 128, 0);
          bulk_wait_all_writes();
        }
        PTRACE_T(128, k, tph, 5);
      }
      ++mma_phase;
    };

    // ---- B1: q, k_s, v_s^T in bf16 from acc_qkv (every CTA a slice) ----------
    auto convert_qkv = [&](int k, int l) {
      const float* cq = a.cqkv + (size_t)(k * L + l) * a.qkvdim;
      const int per_t = a.qkvdim / 8;
      const long total = (long)T * per_t;
      for (long idx = (long)cta * kWork + wt; idx < total; idx += (long)G * kWork) {
        const int t = (int)(idx / per_t), n = (int)(idx - (long)t * per_t) * 8;
        const float rr = __ldcg(a.rms + t);
        const float4 x0 = ldcg4(a.accq + (size_t)t * a.qkvdim + n), x1 = ldcg4(a.accq + (size_t)t * a.qkvdim + n + 4);
        const float4 c0 = __ldg((const float4*)(cq + n)), c1 = __ldg((const float4*)(cq + n + 4));
        const float v[8] = {fmaf(rr, x0.x, c0.x), fmaf(rr, x0.y, c0.y), fmaf(rr, x0.z, c0.z), fmaf(rr, x0.w, c0.w),
                            fmaf(rr, x1.x, c1.x), fmaf(rr, x1.y, c1.y), fmaf(rr, x1.z, c1.z), fmaf(rr, x1.w, c1.w)};
        const int b = t / a.H, i = t - b * a.H;
        if (n < a.qdim) {
          const int j = n / a.d_h, d = n - j * a.d_h;
          __stcg((uint4*)(a.q + (((size_t)b * a.n_q + j) * a.H + i) * a.d_h + d), pack8(v));
        } else if (n < a.qdim + a.kvdim) {
          const int r = n - a.qdim, j = r / a.d_h, d = r - j * a.d_h;
          __stcg((uint4*)(a.ks + (((size_t)b * a.n_kv + j) * a.H + i) * a.d_h + d), pack8(v));
        } else {
          const int r = n - a.qdim - a.kvdim, j = r / a.d_h, d = r - j * a.d_h;
          bf16* dst = a.vs + (((size_t)b * a.n_kv + j) * a.d_h + d) * a.Hp + i;
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[(size_t)e * a.Hp] = __float2bfloat16_rn(v[e]);
        }
      }
    };

    // ---- B2: one attention unit (attention CTAs) ---------------------------------
    auto attention = [&](int unit, int l) {
      const int ch = unit % a.nch;
      int rest = unit / a.nch;
      const int qt = rest % a.nqt;
      rest /= a.nqt;
      const int g = rest % a.n_kv, b = rest / a.n_kv;
      const int rows = a.group * a.H - qt * 128 < 128 ? a.group * a.H - qt * 128 : 128;
      const bool pre = ch < a.npch;                  // a chunk of cached keys or of action keys
      const int k0 = (pre ? ch : ch - a.npch) * kKC; // first key of the chunk in its part
      const int nk_part = pre ? a.P : a.H;
      const int nkeys = nk_part - k0 < kKC ? nk_part - k0 : kKC;
      const int zc = (l * a.B + b) * a.n_kv + g, zs = b * a.n_kv + g;
      const int dh = a.d_h, nsub = dh / 64;
      uint8_t* Qs = smem + As.q;
      uint8_t* Ks = smem + As.k;
      uint8_t* Vt = smem + As.v;
      uint8_t* Ps = smem + As.p;
      const uint32_t tS = tmem + 256u, tO = tmem;
      const uint32_t par = (uint32_t)att_phase & 1u;
      if (threadIdx.x == 32) {
        const uint64_t pol = l2_policy_evict_last();
        fence_proxy_async_global();
        const int qrow = (b * a.n_q + g * a.group) * a.H + qt * 128;
        mbar_arrive_expect_tx(qkbar, 2u * 128u * (uint32_t)dh * 2u);
        for (int s = 0; s < nsub; ++s) {
          tma_load_2d(Qs + (size_t)s * 16384, &m.q, qkbar, s * 64, qrow);
          tma_load_3d_hint(Ks + (size_t)s * 16384, pre ? &m.kc : &m.ks, qkbar, s * 64, k0, pre ? zc : zs, pol);
        }
        mbar_arrive_expect_tx(vbar, 2u * (uint32_t)dh * 128u);
        for (int kh = 0; kh < 2; ++kh)
          tma_load_3d_hint(Vt + (size_t)kh * dh * 128, pre ? &m.vc : &m.vs, vbar, k0 + kh * 64, 0, pre ? zc : zs, pol);
        // S = Q K^T
        if (!mbar_wait(qkbar, par, a.status)) *s_fail = 1;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, kKC);
        for (int s = 0; s < nsub; ++s)
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            umma_bf16(tS, sdesc_k128(smem_u32(Qs + (size_t)s * 16384) + k4 * 32),
                      sdesc_k128(smem_u32(Ks + (size_t)s * 16384) + k4 * 32), idesc, (s > 0 || k4 > 0) ? 1u : 0u);
        umma_commit(sdone);
      }
      if (warp >= 4) {
        // softmax of this unit's rows: one row per thread
        const int row = (warp - 4) * 32 + lane;
        if (!mbar_wait(sdone, par, a.status)) *s_fail = 1;
        tc_fence_after();
        const uint32_t taddr = tS + ((uint32_t)((warp - 4) * 32) << 16);
        float sv[kKC];
#pragma unroll
        for (int q = 0; q < kKC / 16; ++q) tmem_ld16(taddr + (uint32_t)(q * 16), sv + q * 16);
        const bool live = row < rows;
        // visibility of the chunk's keys (prefix chunks under a mask)
        uint32_t mw[4];
        const uint32_t* mrow = (pre && a.pmask) ? a.pmask + (size_t)b * a.pmw : nullptr;
#pragma unroll
        for (int q = 0; q < 4; ++q) mw[q] = prefix_mask_window(mrow, a.pmw, k0 + q * 32);
        auto vis = [&](int j) { return j < nkeys && ((mw[j >> 5] >> (j & 31)) & 1u); };
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < kKC; ++j)
          if (vis(j)) mx = fmaxf(mx, sv[j] * a.scale_log2);
        if (!live) mx = 0.f;
        float lsum = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < kKC / 8; ++c8) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = c8 * 8 + e;
            p[e] = (live && vis(j)) ? fast_exp2(sv[j] * a.scale_log2 - mx) : 0.f;
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
        if (live) __stcg(&a.oml[((size_t)(zs * a.nch + ch)) * (a.group * a.H) + qt * 128 + row], make_float2(mx, lsum));
        fence_proxy_async_smem();
        tc_fence_before();
      }
      named_bar_sync(kBarWork, kWork);
      // O = P V
      if (threadIdx.x == 32) {
        if (!mbar_wait(vbar, par, a.status)) *s_fail = 1;
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
        if (!mbar_wait(odone, par, a.status)) *s_fail = 1;
        tc_fence_after();
        const uint32_t taddr = tO + ((uint32_t)((warp - 4) * 32) << 16);
        float* dst = a.opart + (((size_t)(zs * a.nch + ch)) * (a.group * a.H) + qt * 128 + row) * dh;
        for (int c0 = 0; c0 < dh; c0 += 32) {
          uint32_t r[32];
          tmem_ld16_nowait(taddr + (uint32_t)c0, r);
          tmem_ld16_nowait(taddr + (uint32_t)c0 + 16u, r + 16);
          tmem_wait16(r);
          tmem_wait16(r + 16);
          if (row < rows) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg((uint4*)(dst + c0 + q * 4), make_uint4(r[q * 4], r[q * 4 + 1], r[q * 4 + 2], r[q * 4 + 3]));
          }
        }
        tc_fence_before();
      }
      // the next unit reuses the buffers that P V read: wait for the epilogue
      named_bar_sync(kBarWork, kWork);
      ++att_phase;
    };

    // ---- B3: o = merged chunks (every CTA a slice) -------------------------------
    auto merge = [&]() {
      const int per_t = a.qdim / 8;
      const int GH = a.group * a.H;
      const long total = (long)T * per_t;
      for (long idx = (long)cta * kWork + wt; idx < total; idx += (long)G * kWork) {
        const int t = (int)(idx / per_t), n = (int)(idx - (long)t * per_t) * 8;
        const int j = n / a.d_h, d = n - j * a.d_h;
        const int g = j / a.group, jj = j - g * a.group;
        const int b = t / a.H, i = t - b * a.H;
        const int r = jj * a.H + i;
        const size_t base = (size_t)(b * a.n_kv + g) * a.nch;
        float2 ml[16];
#pragma unroll
        for (int ch = 0; ch < 16; ++ch)
          if (ch < a.nch) ml[ch] = __ldcg(&a.oml[(base + ch) * GH + r]);
        float M = -INFINITY;
#pragma unroll
        for (int ch = 0; ch < 16; ++ch)
          if (ch < a.nch && ml[ch].y > 0.f) M = fmaxf(M, ml[ch].x);
        float den = 0.f, v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
#pragma unroll
        for (int ch = 0; ch < 16; ++ch)
          if (ch < a.nch && ml[ch].y > 0.f) {  // a chunk of hidden keys contributes nothing
            const float w = fast_exp2(ml[ch].x - M);
            den += w * ml[ch].y;
            const float* op = a.opart + ((base + ch) * GH + r) * a.d_h + d;
            const float4 o0 = ldcg4(op), o1 = ldcg4(op + 4);
            v[0] += w * o0.x; v[1] += w * o0.y; v[2] += w * o0.z; v[3] += w * o0.w;
            v[4] += w * o1.x; v[5] += w * o1.y; v[6] += w * o1.z; v[7] += w * o1.w;
          }
        const float inv = 1.f / den;
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] *= inv;
        __stcg((uint4*)(a.o + (size_t)t * a.qdim + n), pack8(v));
      }
    };

    // ---- head, part 1 (every CTA): v[t][o] = W_out[o] . (modulated norm of h[t])
    // and the Euler update; one warp per (token, output) pair, all its loads
    // in flight together --------------------------------------------------------
    auto head_velocity = [&](int k) {
      const float dt = a.dt_sign * (float)((double)(k + 1) / a.S - (double)k / a.S);
      const float* x_in = k == 0 ? a.noise : a.actions;
      const float* gf = a.modf + (size_t)k * 2 * D;
      const float* bf = gf + D;
      const int w7 = warp - 1, nw = G * 7;
      for (int pr = cta * 7 + w7; pr < T * a.d_a; pr += nw) {
        const int t = pr / a.d_a, o = pr - t * a.d_a;
        const float* hr = a.h + (size_t)t * D;
        const float* wo = a.wout + (size_t)o * D;
        float ss = 0.f, dot = 0.f;
        for (int i = lane * 4; i < D; i += 128) {
          const float4 hv = ldcg4(hr + i);
          const float4 g4 = __ldg((const float4*)(gf + i)), w4 = __ldg((const float4*)(wo + i));
          ss += hv.x * hv.x + hv.y * hv.y + hv.z * hv.z + hv.w * hv.w;
          // u = h r (1 + gamma) + beta: the r factor is applied once below
          dot += hv.x * (1.f + g4.x) * w4.x + hv.y * (1.f + g4.y) * w4.y + hv.z * (1.f + g4.z) * w4.z +
                 hv.w * (1.f + g4.w) * w4.w;
        }
        // beta . W_out[o] separately (independent of h)
        float bw = 0.f;
        for (int i = lane * 4; i < D; i += 128) {
          const float4 b4 = __ldg((const float4*)(bf + i)), w4 = __ldg((const float4*)(wo + i));
          bw += b4.x * w4.x + b4.y * w4.y + b4.z * w4.z + b4.w * w4.w;
        }
        ss = warp_sum(ss);
        dot = warp_sum(dot);
        bw = warp_sum(bw);
        if (lane == 0) {
          const float r = rsqrtf(ss / (float)D + a.eps);
          const float v = fmaf(r, dot, bw);
          const size_t idx = (size_t)t * a.d_a + o;
          __stcg(a.actions + idx, fmaf(dt, v, x_in[idx]));
          if (a.vtap) a.vtap[(size_t)k * T * a.d_a + idx] = v;
        }
      }
      if (cta == 0 && wt == 0 && a.abort && *a.abort) {
        latch_error(a.status, VLA_DEV_ABORTED);
        __stcg(a.stop, 1);
      }
    };
    // ---- head, part 2 (every CTA): h[t] = x[t] W_in^T for the next step ---------
    auto head_embed = [&]() {
      const int parts = G / T;  // CTAs per token (T <= GL < G)
      if (cta < parts * T) {
        const int t = cta % T, part = cta / T;
        for (int j = wt; j < a.d_a; j += kWork) xs[j] = __ldcg(a.actions + (size_t)t * a.d_a + j);
        named_bar_sync(kBarWork, kWork);
        const int per = (D + parts - 1) / parts;
        const int i0 = part * per, i1 = i0 + per < D ? i0 + per : D;
        for (int i = i0 + wt; i < i1; i += kWork) {
          const float* w = a.win + (size_t)i * a.d_a;
          float acc = 0.f;
          for (int j = 0; j < a.d_a; ++j) acc += xs[j] * __ldg(w + j);
          __stcg(a.h + (size_t)t * D + i, acc);
        }
        named_bar_sync(kBarWork, kWork);
      }
    };

    // ---- the solve ------------------------------------------------------------
    embed_token(a.noise);
    zero_buf(a.accq, (long)T * a.qkvdim);
    zero_buf(a.accu, (long)T * a.F);
    barrier();
    for (int k = 0; k < a.S && ok; ++k) {
      tk = k;
      tph = 0;
      PTRACE(k, 0, 0);
      for (int l = 0; l < L && ok; ++l) {
        linear(0, k, l);                      // A
        token_rms(a.rms);
        zero_buf(a.accu, (long)T * a.F);
        barrier();
        convert_qkv(k, l);                    // B1
        barrier();
        if (att_cta)                          // B2
          for (int u = cta - GL; u < a.att_units; u += NA) attention(u, l);
        barrier();
        merge();                              // B3
        zero_buf(a.accq, (long)T * a.qkvdim);
        barrier();
        linear(1, k, l);                      // C
        barrier();
        linear(2, k, l);                      // D
        token_rms(a.rms + T);
        barrier();
        linear(3, k, l);                      // E
        barrier();
      }
      if (!ok) break;
      head_velocity(k);
      barrier();
      if (!ok || __ldcg(a.stop)) break;  // abort seen at this step boundary (uniform)
      if (k + 1 < a.S) {
        head_embed();
        barrier();
      }
    }
    if (threadIdx.x == 32) {
      *s_stop = 1;
      // Before TMEM is freed and the CTA exits, every MMA and copy this thread
      // issued must be complete (they are, unless a wait gave up): wait for
      // the last completion of each barrier.
      if (n_mma) {
        mbar_drain(mma_done, (uint32_t)(n_mma - 1) & 1u);
        mbar_drain(bbar, (uint32_t)(n_mma - 1) & 1u);
      }
      if (n_att) {
        mbar_drain(qkbar, (uint32_t)(n_att - 1) & 1u);
        mbar_drain(vbar, (uint32_t)(n_att - 1) & 1u);
        mbar_drain(sdone, (uint32_t)(n_att - 1) & 1u);
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
size_t persist_smem_bytes(int D) {
  (void)D;
  return 1024 + kSmemUse;
}
int persist_ring_stages(int D, int work_bytes) { return persist_layout(D, (uint32_t)work_bytes).R; }
bool persist_att_fits(int dh) { return att_layout(dh).end <= kSmemUse; }

cudaError_t persist_init() { return set_max_dyn_smem(k_solver_persist); }

// CTAs of the kernel that fit on one SM with its shared memory (a
// cooperative launch of one CTA per SM needs 1).
cudaError_t persist_blocks_per_sm(int D, int* n) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k_solver_persist, kThreads, persist_smem_bytes(D));
}

cudaError_t launch_persist(const CUtensorMap* maps, const PersistArgs& a, int grid, cudaStream_t st) {
  const size_t smem = persist_smem_bytes(a.D);
  if (smem > 227 * 1024 || persist_ring_stages(a.D, a.work_bytes) < 4 || !persist_att_fits(a.d_h) || a.n_att < 1 ||
      a.n_att >= grid || a.T > grid - a.n_att || a.nch > 16 || a.d_a > 64)
    return cudaErrorInvalidValue;
  Maps m;
  for (int i = 0; i < 4; ++i) m.w[i] = maps[i];
  m.kc = maps[4]; m.vc = maps[5]; m.ks = maps[6]; m.vs = maps[7]; m.q = maps[8];
  m.hld = maps[9]; m.uld = maps[10]; m.old = maps[11];
  m.red[0] = maps[12]; m.red[1] = maps[13]; m.red[2] = maps[14];
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
  return cudaLaunchKernelEx(&cfg, k_solver_persist, m, a);
}
