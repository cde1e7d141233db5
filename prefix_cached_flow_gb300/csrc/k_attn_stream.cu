// Joint non-causal GQA attention, streaming form ("vla.cpp: A Unified
// Inference Runtime for Vision-Language-Action Models", §III-B Eq. (2)):
//   o = softmax(Q [K_C ; K_s]^T / sqrt(d_h) + M) [V_C ; V_s],  M = 0.
//
// One CTA owns one 128-row query tile of one (observation, K/V head) and
// streams every key through it in 64-key chunks: the cached prefix keys
// first, then the action tokens' own keys.  No partial result leaves the CTA,
// so this form suits many query tiles (batched requests); the clustered
// kernel in k_attn_tc.cu splits one tile's keys over several SMs instead.
//
// Warp roles (352 threads):
//   warps 0-7  softmax and epilogue: warps w and w + 4 share the 32 query
//              rows of TMEM lane quarter w % 4; both read the whole row of
//              S_j and find the same maximum, then warp w exponentiates keys
//              0..31 (and owns the first half of O's columns), warp w + 4
//              keys 32..63 (the second half)
//   warp 8     TMA producer of Q and of K_j (two-stage ring)
//   warp 9     MMA issuer:   S_j = Q K_j^T into one of two TMEM S buffers,
//                            O += P_j V_j into the TMEM O accumulator
//   warp 10    TMA producer of V_j^T (two-stage ring)
// K_j's slot is released when S_j completes and V_j's when P_j V_j does, so
// the key loads run ahead of the softmax.  Per chunk j the softmax thread
// reads its row of S_j, updates the running maximum m, writes
// P_j = exp2(S_j log2e / sqrt(d_h) - m) in bf16 to shared memory and adds it
// to the row sum l.  m is raised lazily: only when a chunk maximum exceeds it
// by more than 2^8 in the exponent are O (in TMEM) and l rescaled, so P never
// exceeds 256 and the final o = O / l is unchanged in exact arithmetic.
// S_{j+1} runs on the tensor cores while P_j is computed; P_j V_j runs while
// S_{j+1} is read.  The output tile is staged in the freed K/V buffers and
// written with row-contiguous stores.
#include "vla_common.cuh"

namespace {

constexpr int KB = 64;              // keys per chunk
constexpr float RESCALE_LOG2 = 8.f; // lazy-rescale threshold (factor 256)

struct StreamSmem {
  uint32_t q, k, v, p, bars, slot, total;
};

// Byte offsets from the 1024-aligned base.  q: nsub x [128][64] bf16;
// k: 2 stages x nsub x [64][64]; v: 2 stages x [d_h][64] (V^T rows);
// p: 2 x [128][64]; every operand tile 128-byte swizzled.
__host__ __device__ inline StreamSmem stream_layout(int d_h) {
  const int nsub = d_h / 64;
  StreamSmem s;
  s.q = 0;
  s.k = s.q + (uint32_t)nsub * 16384u;
  s.v = s.k + 2u * (uint32_t)nsub * 8192u;
  s.p = s.v + 2u * (uint32_t)d_h * 128u;
  s.bars = s.p + 2u * 16384u;
  s.slot = s.bars + 24 * 8;
  s.total = s.slot + 16;
  return s;
}

enum { B_Q = 0, B_KF = 1, B_KE = 3, B_VF = 5, B_VE = 7, B_SF = 9, B_PF = 11, B_PV = 13, B_FIN = 15, B_XL = 16,
       B_ST = 17, B_QT = 18, N_BARS = 19 };
constexpr int NSM = 256;  // softmax threads

__device__ __forceinline__ void tma_load_3d_s(void* dst, const void* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Optional per-CTA cycle stamps (built only with -DVLA_TIMELINE).
#ifdef VLA_TIMELINE
#define TLC(ev)                                                                              \
  do {                                                                                       \
    if (a.tl) a.tl[((size_t)blockIdx.x + gridDim.x * (size_t)blockIdx.y) * 16 + (ev)] = clock64(); \
  } while (0)
#else
#define TLC(ev) \
  do {          \
  } while (0)
#endif

template <bool O32>
__global__ void __launch_bounds__(352, 1)
    k_attn_stream(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ CUtensorMap tmKs,
                  const __grid_constant__ CUtensorMap tmVs, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int dh = a.d_h, nsub = dh / 64;
  const StreamSmem L = stream_layout(dh);
  uint8_t* Qs = smem + L.q;
  uint8_t* Ks = smem + L.k;
  uint8_t* Vs = smem + L.v;
  uint8_t* Ps = smem + L.p;
  uint64_t* bars = (uint64_t*)(smem + L.bars);
  uint32_t* tmem_slot = (uint32_t*)(smem + L.slot);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, bg = blockIdx.y;
  const int b = bg / a.n_kv, gk = bg - b * a.n_kv;
  const int n_pre = (a.P + KB - 1) / KB, n_suf = (a.H + KB - 1) / KB;
  const int nch = n_pre + n_suf;
  // TMEM: O (d_h columns), two S buffers (KB columns each), Q (d_h / 2
  // columns of bf16 pairs: the S MMA reads its A operand from here, not
  // from shared memory, which leaves shared-memory bandwidth to K).
  const uint32_t ncols = dh + 2 * KB + dh / 2 <= 256 ? 256u : 512u;
  const uint32_t s_col = (uint32_t)dh;
  const uint32_t q_col = (uint32_t)(dh + 2 * KB);

  if (threadIdx.x == 0) {
    s_fail = 0;
    mbar_init(&bars[B_Q], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_KF + i], 1);
      mbar_init(&bars[B_KE + i], 1);
      mbar_init(&bars[B_VF + i], 1);
      mbar_init(&bars[B_VE + i], 1);
      mbar_init(&bars[B_SF + i], 1);
      mbar_init(&bars[B_PF + i], NSM);
      mbar_init(&bars[B_PV + i], 1);
    }
    mbar_init(&bars[B_FIN], 1);
    mbar_init(&bars[B_XL], NSM);
    mbar_init(&bars[B_ST], NSM);
    mbar_init(&bars[B_QT], NSM);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (threadIdx.x == 0) TLC(0);

  if (warp == 8 || warp == 10) {
    // ---------------- TMA producers: warp 8 Q and K, warp 10 V^T ----------------
    if (lane == 0) {
      const bool kp = warp == 8;
      const int zc = (a.layer * a.B + b) * a.n_kv + gk;
      const int zs = b * a.n_kv + gk;
      uint64_t* full = &bars[kp ? B_KF : B_VF];
      uint64_t* empty = &bars[kp ? B_KE : B_VE];
      const uint32_t bytes = kp ? (uint32_t)nsub * 8192u : (uint32_t)dh * 128u;
      auto issue = [&](int j) {
        const int st = j & 1;
        mbar_arrive_expect_tx(&full[st], bytes);
        const bool pre = j < n_pre;
        const int k0 = pre ? j * KB : (j - n_pre) * KB;
        if (kp) {
          uint8_t* kd = Ks + (size_t)st * nsub * 8192;
          for (int s = 0; s < nsub; ++s)
            tma_load_3d_s(kd + (size_t)s * 8192, pre ? &tmK : &tmKs, &full[st], s * 64, k0, pre ? zc : zs);
        } else {
          tma_load_3d_s(Vs + (size_t)st * dh * 128, pre ? &tmVt : &tmVs, &full[st], k0, 0, pre ? zc : zs);
        }
      };
      // The cached prefix does not depend on the previous kernel: its first
      // two chunks are in flight before the grid dependency wait.
      int j = 0;
      for (; j < 2 && j < n_pre; ++j) issue(j);
      griddep_wait();
      if (kp) {
        mbar_arrive_expect_tx(&bars[B_Q], (uint32_t)nsub * 16384u);
        const int qrow = (b * a.n_q + gk * a.group) * a.H + qt * 128;
        for (int s = 0; s < nsub; ++s) tma_load_2d(Qs + (size_t)s * 16384, &tmQ, &bars[B_Q], s * 64, qrow);
      }
      for (; j < nch; ++j) {
        if (j >= 2 && !mbar_wait(&empty[j & 1], (uint32_t)((j - 2) >> 1) & 1u, a.status)) {
          s_fail = 1;
          break;
        }

        issue(j);
      }
      // Own copies land before the CTA can exit (normally already consumed).
      const int issued = j;
      for (int i = issued - 2 < 0 ? 0 : issued - 2; i < issued; ++i) mbar_drain(&full[i & 1], (uint32_t)(i >> 1) & 1u);
      if (kp) mbar_drain(&bars[B_Q], 0);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    griddep_wait();
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, KB);
      const uint32_t idesc_o = idesc_bf16_f32(128, dh);
      bool ok = mbar_wait(&bars[B_QT], 0, a.status);
      auto pv = [&](int i) -> bool {
        const int st = i & 1;
        if (!mbar_wait(&bars[B_PF + st], (uint32_t)(i >> 1) & 1u, a.status)) return false;

        if (!mbar_wait(&bars[B_VF + st], (uint32_t)(i >> 1) & 1u, a.status)) return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(Ps + (size_t)st * 16384), va = smem_u32(Vs + (size_t)st * dh * 128);
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk)
          umma_bf16(tmem, sdesc_k128(pa + kk * 32), sdesc_k128(va + kk * 32), idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars[B_PV + st]);
        umma_commit(&bars[B_VE + st]);
        return true;
      };
      int j = 0;
      for (; ok && j < nch; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&bars[B_KF + st], (uint32_t)(j >> 1) & 1u, a.status)) {
          ok = false;
          break;
        }

        tc_fence_after();
        const uint32_t ka = smem_u32(Ks + (size_t)st * nsub * 8192);
        for (int s = 0; s < nsub; ++s) {
          const uint32_t kb = ka + (uint32_t)s * 8192u;
#pragma unroll
          for (int k = 0; k < 4; ++k)  // K step of 16 = 8 TMEM columns of Q
            umma_bf16_ts(tmem + s_col + (uint32_t)(st * KB), tmem + q_col + (uint32_t)((s * 4 + k) * 8),
                         sdesc_k128(kb + k * 32), idesc_s, (s > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_SF + st]);
        umma_commit(&bars[B_KE + st]);
        if (j >= 1 && !pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) ok = pv(nch - 1);
      if (!ok) s_fail = 1;
      // Every MMA issued above has completed before TMEM is freed.
      umma_commit(&bars[B_FIN]);
      mbar_drain(&bars[B_FIN], 0);

    }
    __syncwarp();
  } else {
    // ---------------- softmax + epilogue (warps 0-7) ----------------
    griddep_wait();
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;  // query row in the tile = TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const int hc = dh / 2;                // O columns of this half
    float m_used = -INFINITY, l = 0.f;
    bool ok = __all_sync(~0u, mbar_wait(&bars[B_Q], 0, a.status));
    // Q row into TMEM (the S MMA's A operand): groups of four 16-byte chunks
    // (32 bf16 = 16 columns) read from the 128-byte-swizzled shared tile;
    // the two warps of a lane quarter take half of the groups each.
    if (ok) {
      const int G = nsub * 2;
      for (int gi = half * G / 2; gi < (half + 1) * G / 2; ++gi) {
        const uint8_t* rowp = Qs + (size_t)(gi >> 1) * 16384 + (size_t)row * 128;
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t j = (uint32_t)((gi & 1) * 4 + q);
          const uint4 u = *(const uint4*)(rowp + ((j ^ (uint32_t)(row & 7)) << 4));
          w[q * 4 + 0] = u.x;
          w[q * 4 + 1] = u.y;
          w[q * 4 + 2] = u.z;
          w[q * 4 + 3] = u.w;
        }
        tmem_st16(trow + q_col + (uint32_t)(gi * 16), w);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    mbar_arrive(&bars[B_QT]);
    for (int j = 0; ok && j < nch; ++j) {
      const int st = j & 1;
      if (!__all_sync(~0u, mbar_wait(&bars[B_SF + st], (uint32_t)(j >> 1) & 1u, a.status))) {
        ok = false;
        break;
      }
      if (row == 0 && half == 0) {
      }
      tc_fence_after();
      const int nk = j < n_pre ? (a.P - j * KB < KB ? a.P - j * KB : KB)
                               : (a.H - (j - n_pre) * KB < KB ? a.H - (j - n_pre) * KB : KB);
      const int nkh = nk - half * 32;  // valid keys in this half (may be <= 0)
      uint32_t sr[KB];
#pragma unroll
      for (int q = 0; q < KB / 16; ++q) tmem_ld16_nowait(trow + s_col + (uint32_t)(st * KB + q * 16), sr + q * 16);
#pragma unroll
      for (int q = 0; q < KB / 16; ++q) tmem_wait16(sr + q * 16);
      // Row maximum over all keys of the chunk (both warps of the pair reach
      // the same value; eight independent chains; the scale is positive, so
      // it is applied once).
      float mxv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mxv[u] = -INFINITY;
      if (nk == KB) {  // full chunk (all but the last prefix and the action chunk): no masks
#pragma unroll
        for (int u = 0; u < KB; ++u) mxv[u & 7] = fmaxf(mxv[u & 7], __uint_as_float(sr[u]));
      } else {
#pragma unroll
        for (int u = 0; u < KB; ++u) mxv[u & 7] = fmaxf(mxv[u & 7], u < nk ? __uint_as_float(sr[u]) : -INFINITY);
      }
      const float mx = fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                             fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7]))) * a.scale_log2;
      // The decision is per warp (tcgen05.ld / st are warp-collective) and the
      // two warps of a pair see the same rows, maxima and history, so they
      // decide alike; a row whose maximum did not grow scales by 1.
      if (__any_sync(~0u, mx > m_used + RESCALE_LOG2)) {
        const float m_new = fmaxf(m_used, mx);
        if (j > 0) {
          // O holds sum_{i<j} P_i V_i at the old maximum: wait for the last
          // product, then scale this half of the row by 2^(m_used - m_new).
          if (!__all_sync(~0u, mbar_wait(&bars[B_PV + ((j - 1) & 1)], (uint32_t)((j - 1) >> 1) & 1u, a.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = fast_exp2(m_used - m_new);
          for (int c0 = half * hc; c0 < (half + 1) * hc; c0 += 32) {
            uint32_t r[32];
            tmem_ld16_nowait(trow + (uint32_t)c0, r);
            tmem_ld16_nowait(trow + (uint32_t)(c0 + 16), r + 16);
            tmem_wait16(r);
            tmem_wait16(r + 16);
#pragma unroll
            for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * f);
            tmem_st16(trow + (uint32_t)c0, r);
            tmem_st16(trow + (uint32_t)(c0 + 16), r + 16);
          }
          tmem_wait_st();
          l *= f;
        }
        m_used = m_new;
      }
      // P buffer st is free once P_{j-2} V_{j-2} has completed.
      if (j >= 2 && !__all_sync(~0u, mbar_wait(&bars[B_PV + st], (uint32_t)((j - 2) >> 1) & 1u, a.status))) {
        ok = false;
        break;
      }
      const uint32_t pa = smem_u32(Ps + (size_t)st * 16384);
      const float nm = -m_used;
      uint32_t sh[32];  // this half's keys (register selects, no indexed array)
#pragma unroll
      for (int u = 0; u < 32; ++u) sh[u] = half ? sr[32 + u] : sr[u];
      float lv[4] = {0.f, 0.f, 0.f, 0.f};
      const bool full = nkh >= 32;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float p[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = q * 8 + u;
          p[u] = fast_exp2(fmaf(__uint_as_float(sh[c]), a.scale_log2, nm));
          if (!full) p[u] = c < nkh ? p[u] : 0.f;
          lv[u & 3] += p[u];
        }
        uint4 pk;
        pk.x = pack_bf16x2(p[0], p[1]);
        pk.y = pack_bf16x2(p[2], p[3]);
        pk.z = pack_bf16x2(p[4], p[5]);
        pk.w = pack_bf16x2(p[6], p[7]);
        st_shared_v4_u32(pa + sw128_offset((uint32_t)row, (uint32_t)(half * 4 + q)), pk);
      }
      l += (lv[0] + lv[1]) + (lv[2] + lv[3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[B_PF + st]);
    }
    if (!ok) s_fail = 1;
    // Epilogue: o = O / l with l the sum of the pair's partial sums.  Each
    // thread stages its half of the row (scaled, in the output type) in the
    // K/V buffers, which every MMA and copy has finished with, 16-byte chunks
    // XOR-swizzled by row; then each warp writes whole rows with consecutive
    // lanes on consecutive 16-byte chunks.  All waits are bounded.
    const bool fin =
        ok && __all_sync(~0u, mbar_wait(&bars[B_PV + ((nch - 1) & 1)], (uint32_t)((nch - 1) >> 1) & 1u, a.status));
    constexpr int ES = O32 ? 4 : 2;     // output element size
    const int RB = dh * ES;             // bytes per staged row
    const int NC = RB / 16;             // 16-byte chunks per row (8..64)
    const uint32_t stage = smem_u32(Ks);
    float* xl = (float*)Ps;  // [2][128] partial row sums (the P buffers are free now)
    xl[half * 128 + row] = l;
    mbar_arrive(&bars[B_XL]);
    const bool lok = __all_sync(~0u, mbar_wait(&bars[B_XL], 0, a.status));
    const int nrows = (a.group * a.H - qt * 128) < 128 ? (a.group * a.H - qt * 128) : 128;
    uint8_t* obytes = O32 ? (uint8_t*)a.o32 : (uint8_t*)a.o;
    uint8_t** orows = (uint8_t**)(Ps + 1024);  // [128] output row addresses (P buffers are free)
    if (half == 0) {
      const int rg = qt * 128 + row;  // (query head within the group, action token)
      const int jj = rg / a.H, i = rg - jj * a.H;
      orows[row] = obytes + (((size_t)b * a.H + i) * (size_t)(a.n_q * dh) + (size_t)(gk * a.group + jj) * dh) * ES;
    }
    if (fin && lok) {
      tc_fence_after();
      const float inv = 1.f / (xl[row] + xl[128 + row]);
      const uint32_t rbase = stage + (uint32_t)(row * RB);
      for (int c0 = half * hc; c0 < (half + 1) * hc; c0 += 32) {
        uint32_t r[32];
        tmem_ld16_nowait(trow + (uint32_t)c0, r);
        tmem_ld16_nowait(trow + (uint32_t)(c0 + 16), r + 16);
        tmem_wait16(r);
        tmem_wait16(r + 16);
        if (O32) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int c = c0 / 4 + q;  // chunk index within the row
            uint4 u = make_uint4(__float_as_uint(__uint_as_float(r[4 * q]) * inv),
                                 __float_as_uint(__uint_as_float(r[4 * q + 1]) * inv),
                                 __float_as_uint(__uint_as_float(r[4 * q + 2]) * inv),
                                 __float_as_uint(__uint_as_float(r[4 * q + 3]) * inv));
            st_shared_v4_u32(rbase + (uint32_t)(((c ^ row) & (NC - 1)) * 16), u);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = c0 / 8 + q;
            const uint32_t* w = r + q * 8;
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv);
            u.y = pack_bf16x2(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv);
            u.z = pack_bf16x2(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv);
            u.w = pack_bf16x2(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv);
            st_shared_v4_u32(rbase + (uint32_t)(((c ^ row) & (NC - 1)) * 16), u);
          }
        }
      }
    }
    mbar_arrive(&bars[B_ST]);
    const bool sok = __all_sync(~0u, mbar_wait(&bars[B_ST], 0, a.status));
    if (sok && s_fail == 0) {
      // Warp w copies rows w, w + 8, ... (NC >= 32: a row per pass, lanes on
      // consecutive 16-byte chunks) or 32 / NC rows per pass (NC < 32).
      const int rpi = NC >= 32 ? 1 : 32 / NC;   // rows per warp pass
      const int cpl = NC >= 32 ? NC / 32 : 1;   // chunks per lane
      const int sub = NC >= 32 ? 0 : lane / NC, cl = NC >= 32 ? lane : lane % NC;
      const uint8_t* sbase = Ks;
#pragma unroll 4
      for (int r0 = warp * rpi; r0 < nrows; r0 += 8 * rpi) {
        const int r = r0 + sub;
        if (r < nrows) {
          uint8_t* orow = orows[r];
          for (int k = 0; k < cpl; ++k) {
            const int c = cl + k * 32;
            *(uint4*)(orow + (size_t)c * 16) = *(const uint4*)(sbase + r * RB + ((c ^ r) & (NC - 1)) * 16);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) TLC(11);
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

}  // namespace

size_t attn_stream_smem_bytes(int d_h) { return 1024 + stream_layout(d_h).total; }

cudaError_t attn_stream_init() {
  cudaError_t e = set_max_dyn_smem(k_attn_stream<false>);
  if (e == cudaSuccess) e = set_max_dyn_smem(k_attn_stream<true>);
  return e;
}

cudaError_t launch_attn_stream(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmVt,
                               const CUtensorMap* tmKs, const CUtensorMap* tmVs, const AttnArgs& a, cudaStream_t st) {
  if ((a.d_h != 64 && a.d_h != 128 && a.d_h != 256) || a.P < 1 || a.H < 1 || a.n_qt < 1 ||
      a.n_qt * 128 < a.group * a.H)
    return cudaErrorInvalidValue;
  const size_t smem = attn_stream_smem_bytes(a.d_h);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_qt, a.B * a.n_kv, 1);
  cfg.blockDim = dim3(352, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.o32) return cudaLaunchKernelEx(&cfg, k_attn_stream<true>, *tmQ, *tmK, *tmVt, *tmKs, *tmVs, a);
  return cudaLaunchKernelEx(&cfg, k_attn_stream<false>, *tmQ, *tmK, *tmVt, *tmKs, *tmVs, a);
}
