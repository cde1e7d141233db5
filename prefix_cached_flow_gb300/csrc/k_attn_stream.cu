// Joint non-causal GQA attention, streaming form ("vla.cpp: A Unified
// Inference Runtime for Vision-Language-Action Models", §III-B Eq. (2)):
//   o = softmax(Q [K_C ; K_s]^T / sqrt(d_h) + M) [V_C ; V_s],  M = 0.
//
// One CTA owns one 128-row query tile of one (observation, K/V head) and
// streams every key through it in 128-key chunks: the cached prefix keys
// first, then the action tokens' own keys.  No partial result leaves the CTA,
// so this form suits many query tiles (batched requests); the clustered
// kernel in k_attn_tc.cu splits one tile's keys over several SMs instead.
//
// One thread feeds the tensor cores one MMA instruction at a time, and an
// instruction costs about the same to issue for any N up to 128, so a chunk
// is 128 keys: S_j = Q K_j^T is d_h / 16 MMAs of N = 128.  Q lives in TMEM
// (the S MMA's A operand); TMEM holds O, Q and one S buffer.  Shared memory
// holds a ring of three chunk slots and one P tile: a slot receives K_j, and
// once S_j is done, V_j^T in its place, so V_j streams in while the softmax
// of chunk j runs, and K_{j+3} follows once P_j V_j is done.
//
// Warp roles (352 threads):
//   warps 0-7  softmax and epilogue: warps w and w + 4 share the 32 query
//              rows of TMEM lane quarter w % 4; both read the whole row of
//              S_j and find the same maximum, then warp w exponentiates keys
//              0..63 of the chunk (and owns the first half of O's columns),
//              warp w + 4 keys 64..127 (the second half)
//   warp 8     TMA producer of Q and of K_j
//   warp 9     MMA issuer: S_j into the TMEM S buffer, O += P_j V_j into the
//              TMEM O accumulator
//   warp 10    TMA producer of V_j^T
// Per chunk j a softmax thread copies its half of its row of S_j into
// registers while finding the row maximum over the whole chunk, then
// releases the S buffer (the next chunk's S MMAs start while it works),
// updates the running maximum m, writes P_j = exp2(S_j log2e / sqrt(d_h) - m)
// in bf16 to shared memory and adds it to the row sum l.  m is raised lazily:
// only when a chunk maximum exceeds it by more than 2^8 in the exponent are O
// (in TMEM) and l rescaled, so P never exceeds 256 and the final o = O / l is
// unchanged in exact arithmetic.  The output tile is staged in the freed
// slots and written one bulk copy per row.
#include "vla_common.cuh"

namespace {

constexpr int KB = 128;              // keys per chunk
constexpr float RESCALE_LOG2 = 8.f;  // lazy-rescale threshold (factor 256)

constexpr int NSLOT = 3;              // chunk slots in the ring

struct StreamSmem {
  uint32_t kv, slot_bytes, p, bars, tslot, total;
};

// Byte offsets from the 1024-aligned base, every operand tile 128-byte
// swizzled.  kv: NSLOT slots of d_h x 256 bytes, each holding either K_j
// (nsub x [128 keys][64]) or V_j^T (2 x [d_h][64 keys], the chunk's two
// 64-key halves); slot 2 first holds Q (nsub x [128 rows][64]) until Q is in
// TMEM.  p: 2 x [128][64 keys].
__host__ __device__ inline StreamSmem stream_layout(int d_h) {
  StreamSmem s;
  s.kv = 0;
  s.slot_bytes = (uint32_t)d_h * 256u;
  s.p = s.kv + NSLOT * s.slot_bytes;
  s.bars = s.p + 2u * 16384u;
  s.tslot = s.bars + 24 * 8;
  s.total = s.tslot + 16;
  return s;
}

enum {
  B_Q = 0,     // Q landed in slot 2
  B_QT = 1,    // Q copied into TMEM (count NSM)
  B_FK = 2,    // [NSLOT] K_j landed in its slot
  B_FV = 5,    // [NSLOT] V_j^T landed in its slot
  B_ES = 8,    // [NSLOT] S_j done: the slot may take V_j^T
  B_EP = 11,   // [NSLOT] P_j V_j done: the slot is free
  B_SF = 14,   // S ready (MMA commit)
  B_SC = 15,   // S read by every softmax thread (count NSM)
  B_PF = 16,   // P tile written (count NSM)
  B_PV = 17,   // P V done (MMA commit)
  B_FIN = 18,  // every MMA of the CTA complete
  B_XL = 19,   // row-sum halves exchanged (count NSM)
  B_ST = 20,   // output tile staged (count NSM)
  N_BARS = 21
};
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

// Row maximum of 32 S values; with MASK only keys (base + u) below nk count.
// The unmasked form uses the three-input max (two new values per op).
// Word j / 32 of a chunk's four visibility words, by selects (no local memory).
__device__ __forceinline__ uint32_t mword(const uint32_t* mw, int j) {
  const int q = j >> 5;
  return q == 0 ? mw[0] : (q == 1 ? mw[1] : (q == 2 ? mw[2] : mw[3]));
}

template <bool MASK>
__device__ __forceinline__ void max32(float (&mx)[4], const uint32_t* r, int base, int nk, const uint32_t* mw) {
  if (MASK) {
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int j = base + u;
      const bool v = j < nk && ((mword(mw, j) >> (j & 31)) & 1u);
      mx[u & 3] = fmaxf(mx[u & 3], v ? __uint_as_float(r[u]) : -INFINITY);
    }
  } else {
#pragma unroll
    for (int u = 0; u < 32; u += 2) {
      float& m = mx[(u >> 1) & 3];
      asm("max.f32 %0, %0, %1, %2;" : "+f"(m) : "f"(__uint_as_float(r[u])), "f"(__uint_as_float(r[u + 1])));
    }
  }
}

__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Probabilities of 64 keys (this half of a row), p = 2^(s * c - m), packed in
// bf16 pairs into pk, their fp32 sum returned.  Without MASK every key is
// valid (a full chunk) and the scale and the sum run on fp32 pairs.
template <bool MASK>
__device__ __forceinline__ float probs64(const uint32_t* sr, uint32_t* pk, float c, float nm, int base, int nk,
                                         const uint32_t* mw) {
  if (MASK) {
    float lv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 64; u += 2) {
      float p0 = fast_exp2(fmaf(__uint_as_float(sr[u]), c, nm));
      float p1 = fast_exp2(fmaf(__uint_as_float(sr[u + 1]), c, nm));
      const int j0 = base + u, j1 = j0 + 1;
      p0 = (j0 < nk && ((mword(mw, j0) >> (j0 & 31)) & 1u)) ? p0 : 0.f;
      p1 = (j1 < nk && ((mword(mw, j1) >> (j1 & 31)) & 1u)) ? p1 : 0.f;
      lv[u & 3] += p0;
      lv[(u + 1) & 3] += p1;
      pk[u >> 1] = pack_bf16x2(p0, p1);
    }
    return (lv[0] + lv[1]) + (lv[2] + lv[3]);
  }
  const uint64_t c2 = f32x2(c, c), n2 = f32x2(nm, nm);
  uint64_t acc[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
  for (int u = 0; u < 64; u += 2) {
    uint64_t x2;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x2) : "l"(f32x2(__uint_as_float(sr[u]), __uint_as_float(sr[u + 1]))),
        "l"(c2), "l"(n2));
    float x0, x1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(x2));
    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc[(u >> 1) & 1]) : "l"(f32x2(p0, p1)));
    pk[u >> 1] = pack_bf16x2(p0, p1);
  }
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc[0]) : "l"(acc[1]));
  float a0, a1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc[0]));
  return a0 + a1;
}

template <bool O32, bool MASKED>
__global__ void __launch_bounds__(352, 1)
    k_attn_stream(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ CUtensorMap tmKs,
                  const __grid_constant__ CUtensorMap tmVs, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int dh = a.d_h, nsub = dh / 64;
  const StreamSmem L = stream_layout(dh);
  uint8_t* KV = smem + L.kv;
  const uint32_t SB = L.slot_bytes;
  uint8_t* Qs = KV + 2 * (size_t)SB;  // slot 2 holds Q first
  uint8_t* Ps = smem + L.p;
  uint64_t* bars = (uint64_t*)(smem + L.bars);
  uint32_t* tmem_slot = (uint32_t*)(smem + L.tslot);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, bg = blockIdx.y;
  const int b = bg / a.n_kv, gk = bg - b * a.n_kv;
  const int n_pre = (a.P + KB - 1) / KB, n_suf = a.no_suffix ? 0 : (a.H + KB - 1) / KB;  // cross layers: none
  const int nch = n_pre + n_suf;
  // TMEM: O (d_h columns), S (KB columns), Q (d_h / 2 columns of bf16 pairs).
  const uint32_t ncols = dh + KB + dh / 2 <= 256 ? 256u : 512u;
  const uint32_t s_col = (uint32_t)dh;
  const uint32_t q_col = (uint32_t)(dh + KB);

  if (threadIdx.x == 0) {
    s_fail = 0;
    mbar_init(&bars[B_Q], 1);
    mbar_init(&bars[B_QT], NSM);
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&bars[B_FK + i], 1);
      mbar_init(&bars[B_FV + i], 1);
      mbar_init(&bars[B_ES + i], 1);
      mbar_init(&bars[B_EP + i], 1);
    }
    mbar_init(&bars[B_SF], 1);
    mbar_init(&bars[B_SC], NSM);
    mbar_init(&bars[B_PF], NSM);
    mbar_init(&bars[B_PV], 1);
    mbar_init(&bars[B_FIN], 1);
    mbar_init(&bars[B_XL], NSM);
    mbar_init(&bars[B_ST], NSM);
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
      auto issue = [&](int j) {
        const bool pre = j < n_pre;
        const int k0 = pre ? j * KB : (j - n_pre) * KB;
        const int sl = j % NSLOT;
        uint8_t* dst = KV + (size_t)sl * SB;
        if (kp) {
          uint64_t* fb = &bars[B_FK + sl];
          mbar_arrive_expect_tx(fb, SB);
          for (int t = 0; t < nsub; ++t)
            tma_load_3d_s(dst + (size_t)t * 16384, pre ? &tmK : &tmKs, fb, t * 64, k0, pre ? zc : zs);
        } else {
          uint64_t* fb = &bars[B_FV + sl];
          mbar_arrive_expect_tx(fb, SB);
          for (int hh = 0; hh < 2; ++hh)
            tma_load_3d_s(dst + (size_t)hh * dh * 128, pre ? &tmVt : &tmVs, fb, k0 + hh * 64, 0, pre ? zc : zs);
        }
      };
      // The cached prefix does not depend on the previous kernel: its first
      // two K chunks are in flight before the grid dependency wait.
      int j = 0;
      if (kp)
        for (; j < 2 && j < n_pre; ++j) issue(j);
      griddep_wait();
      if (kp) {
        mbar_arrive_expect_tx(&bars[B_Q], (uint32_t)nsub * 16384u);
        const int qrow = (b * a.n_q + gk * a.group) * a.H + qt * 128;
        for (int t = 0; t < nsub; ++t) tma_load_2d(Qs + (size_t)t * 16384, &tmQ, &bars[B_Q], t * 64, qrow);
      }
      for (; j < nch; ++j) {
        const int sl = j % NSLOT;
        bool w = true;
        if (kp) {
          // K_j: slot 2 first holds Q; later a slot is free once P_{j-3} V_{j-3} is done.
          if (j == 2) w = mbar_wait(&bars[B_QT], 0, a.status);
          else if (j >= NSLOT) w = mbar_wait(&bars[B_EP + sl], (uint32_t)(j / NSLOT - 1) & 1u, a.status);
        } else {
          w = mbar_wait(&bars[B_ES + sl], (uint32_t)(j / NSLOT) & 1u, a.status);  // V_j^T replaces K_j
        }
        if (!w) {
          s_fail = 1;
          break;
        }
        issue(j);
      }
      // Own copies land before the CTA can exit (normally already consumed):
      // the last use of each slot.
      for (int i = j - NSLOT < 0 ? 0 : j - NSLOT; i < j; ++i)
        mbar_drain(&bars[(kp ? B_FK : B_FV) + i % NSLOT], (uint32_t)(i / NSLOT) & 1u);
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
        const int sl = i % NSLOT;
        if (!mbar_wait(&bars[B_PF], (uint32_t)i & 1u, a.status)) return false;
        if (!mbar_wait(&bars[B_FV + sl], (uint32_t)(i / NSLOT) & 1u, a.status)) return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(Ps), va = smem_u32(KV + (size_t)sl * SB);
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk) {
          const uint32_t hp = (uint32_t)(kk >> 2), ko = (uint32_t)(kk & 3) * 32u;
          umma_bf16(tmem, sdesc_k128(pa + hp * 16384u + ko), sdesc_k128(va + hp * (uint32_t)dh * 128u + ko), idesc_o,
                    (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_PV]);
        umma_commit(&bars[B_EP + sl]);
        return true;
      };
      for (int j = 0; ok && j < nch; ++j) {
        const int sl = j % NSLOT;
        if (!mbar_wait(&bars[B_FK + sl], (uint32_t)(j / NSLOT) & 1u, a.status) ||
            (j >= 1 && !mbar_wait(&bars[B_SC], (uint32_t)(j - 1) & 1u, a.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ka = smem_u32(KV + (size_t)sl * SB);
        for (int s = 0; s < nsub; ++s) {
          const uint32_t kb = ka + (uint32_t)s * 16384u;
#pragma unroll
          for (int k = 0; k < 4; ++k)  // K step of 16 = 8 TMEM columns of Q
            umma_bf16_ts(tmem + s_col, tmem + q_col + (uint32_t)((s * 4 + k) * 8), sdesc_k128(kb + k * 32), idesc_s,
                         (s > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_SF]);
        umma_commit(&bars[B_ES + sl]);
        if (j >= 1 && !pv(j - 1)) ok = false;
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
    const int own0 = half * 64, oth0 = 64 - own0;  // this half's keys / the other half's, within a chunk
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
          const uint32_t jq = (uint32_t)((gi & 1) * 4 + q);
          const uint4 u = *(const uint4*)(rowp + ((jq ^ (uint32_t)(row & 7)) << 4));
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
      if (!__all_sync(~0u, mbar_wait(&bars[B_SF], (uint32_t)j & 1u, a.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int nk = j < n_pre ? (a.P - j * KB < KB ? a.P - j * KB : KB)
                               : (a.H - (j - n_pre) * KB < KB ? a.H - (j - n_pre) * KB : KB);
      // This half's 64 scores stay in registers; the other half is read for
      // the maximum only.  Both warps of a pair reach the same maximum.
      uint32_t sr[64], ot[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld16_nowait(trow + s_col + (uint32_t)(own0 + q * 16), sr + q * 16);
      tmem_ld16_nowait(trow + s_col + (uint32_t)oth0, ot);
      tmem_ld16_nowait(trow + s_col + (uint32_t)(oth0 + 16), ot + 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_wait16(sr + q * 16);
      tmem_wait16(ot);
      tmem_wait16(ot + 16);
      // visibility of the chunk's 128 keys (prefix chunks under a mask)
      // (a separate instantiation: without a mask this costs nothing)
      uint32_t mw[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
      if (MASKED && j < n_pre) {
        const uint32_t* mrow = a.pmask + (size_t)b * a.pmw;
#pragma unroll
        for (int q = 0; q < 4; ++q) mw[q] = prefix_mask_window(mrow, a.pmw, j * KB + q * 32);
      }
      const bool fullc = nk == KB && (!MASKED || (mw[0] & mw[1] & mw[2] & mw[3]) == 0xFFFFFFFFu);  // CTA-uniform
      float mxv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (fullc) {
        max32<false>(mxv, sr, 0, 0, mw);
        max32<false>(mxv, sr + 32, 0, 0, mw);
        max32<false>(mxv, ot, 0, 0, mw);
      } else {
        max32<true>(mxv, sr, own0, nk, mw);
        max32<true>(mxv, sr + 32, own0 + 32, nk, mw);
        max32<true>(mxv, ot, oth0, nk, mw);
      }
      tmem_ld16_nowait(trow + s_col + (uint32_t)(oth0 + 32), ot);
      tmem_ld16_nowait(trow + s_col + (uint32_t)(oth0 + 48), ot + 16);
      tmem_wait16(ot);
      tmem_wait16(ot + 16);
      if (fullc) max32<false>(mxv, ot, 0, 0, mw);
      else max32<true>(mxv, ot, oth0 + 32, nk, mw);
      // S is no longer needed: the next chunk's S MMAs may overwrite it.
      tc_fence_before();
      mbar_arrive(&bars[B_SC]);
      const float mx = fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])) * a.scale_log2;  // scale > 0
      // The decision is per warp (tcgen05.ld / st are warp-collective) and the
      // two warps of a pair see the same rows, maxima and history, so they
      // decide alike; a row whose maximum did not grow scales by 1.
      bool waited_pv = false;
      if (__any_sync(~0u, mx > m_used + RESCALE_LOG2)) {
        const float m_new = fmaxf(m_used, mx);
        if (j > 0) {
          // O holds sum_{i<j} P_i V_i at the old maximum: wait for the last
          // product, then scale this half of the row by 2^(m_used - m_new).
          if (!__all_sync(~0u, mbar_wait(&bars[B_PV], (uint32_t)(j - 1) & 1u, a.status))) {
            ok = false;
            break;
          }
          waited_pv = true;
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
      // Probabilities of this half's 64 keys, packed in bf16 pairs.
      const float nm = -m_used;
      uint32_t pk[32];
      l += fullc ? probs64<false>(sr, pk, a.scale_log2, nm, 0, 0, mw)
                 : probs64<true>(sr, pk, a.scale_log2, nm, own0, nk, mw);
      // The P tile is free once P_{j-1} V_{j-1} has completed.
      if (j >= 1 && !waited_pv && !__all_sync(~0u, mbar_wait(&bars[B_PV], (uint32_t)(j - 1) & 1u, a.status))) {
        ok = false;
        break;
      }
      const uint32_t pa = smem_u32(Ps) + (uint32_t)half * 16384u;  // this half's keys: one 128-byte row
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4_u32(pa + sw128_offset((uint32_t)row, (uint32_t)q),
                         make_uint4(pk[q * 4], pk[q * 4 + 1], pk[q * 4 + 2], pk[q * 4 + 3]));
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[B_PF]);
    }
    if (!ok) s_fail = 1;
    // Epilogue: o = O / l with l the sum of the pair's partial sums.  Each
    // thread stages its half of the row (scaled, in the output type) in the
    // chunk slots, which every MMA and copy has finished with: rows of
    // d_h elements, 16 bytes apart beyond their length so that the 32 rows of
    // a warp's store fall in different banks.  Each row is then one bulk copy
    // to its place in o, issued by the thread that owns the row.  All waits
    // are bounded.
    const bool fin =
        ok && __all_sync(~0u, mbar_wait(&bars[B_PV], (uint32_t)(nch - 1) & 1u, a.status));
    constexpr int ES = O32 ? 4 : 2;     // output element size
    const int RB = dh * ES;             // bytes per output row
    const int RP = RB + 16;             // staged row pitch (128 rows fit in the slots)
    const uint32_t stage = smem_u32(KV);
    float* xl = (float*)Ps;  // [2][128] partial row sums (the P tile is free now)
    xl[half * 128 + row] = l;
    mbar_arrive(&bars[B_XL]);
    const bool lok = __all_sync(~0u, mbar_wait(&bars[B_XL], 0, a.status));
    const int nrows = (a.group * a.H - qt * 128) < 128 ? (a.group * a.H - qt * 128) : 128;
    const uint32_t rbase = stage + (uint32_t)(row * RP);
    if (fin && lok) {
      tc_fence_after();
      const float inv = 1.f / (xl[row] + xl[128 + row]);
      for (int c0 = half * hc; c0 < (half + 1) * hc; c0 += 32) {
        uint32_t r[32];
        tmem_ld16_nowait(trow + (uint32_t)c0, r);
        tmem_ld16_nowait(trow + (uint32_t)(c0 + 16), r + 16);
        tmem_wait16(r);
        tmem_wait16(r + 16);
        if (O32) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint4 u = make_uint4(__float_as_uint(__uint_as_float(r[4 * q]) * inv),
                                 __float_as_uint(__uint_as_float(r[4 * q + 1]) * inv),
                                 __float_as_uint(__uint_as_float(r[4 * q + 2]) * inv),
                                 __float_as_uint(__uint_as_float(r[4 * q + 3]) * inv));
            st_shared_v4_u32(rbase + (uint32_t)((c0 / 4 + q) * 16), u);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t* w = r + q * 8;
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv);
            u.y = pack_bf16x2(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv);
            u.z = pack_bf16x2(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv);
            u.w = pack_bf16x2(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv);
            st_shared_v4_u32(rbase + (uint32_t)((c0 / 8 + q) * 16), u);
          }
        }
      }
    }
    fence_proxy_async_smem();  // the staged rows are read by the bulk copies
    mbar_arrive(&bars[B_ST]);
    const bool sok = __all_sync(~0u, mbar_wait(&bars[B_ST], 0, a.status));
    if (half == 0 && sok && s_fail == 0 && row < nrows) {
      const int rg = qt * 128 + row;  // (query head within the group, action token)
      const int jj = rg / a.H, i = rg - jj * a.H;
      uint8_t* orow = (O32 ? (uint8_t*)a.o32 : (uint8_t*)a.o) +
                      (((size_t)b * a.H + i) * (size_t)(a.n_q * dh) + (size_t)(gk * a.group + jj) * dh) * ES;
      bulk_store_s2g(orow, rbase, (uint32_t)RB);
      bulk_commit_wait_read();
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
  cudaError_t e = set_max_dyn_smem(k_attn_stream<false, false>);
  if (e == cudaSuccess) e = set_max_dyn_smem(k_attn_stream<true, false>);
  if (e == cudaSuccess) e = set_max_dyn_smem(k_attn_stream<false, true>);
  if (e == cudaSuccess) e = set_max_dyn_smem(k_attn_stream<true, true>);
  return e;
}

// The K maps (prefix and action keys) must have 128-row boxes here.
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
  if (a.pmask) {
    if (a.o32) return cudaLaunchKernelEx(&cfg, k_attn_stream<true, true>, *tmQ, *tmK, *tmVt, *tmKs, *tmVs, a);
    return cudaLaunchKernelEx(&cfg, k_attn_stream<false, true>, *tmQ, *tmK, *tmVt, *tmKs, *tmVs, a);
  }
  if (a.o32) return cudaLaunchKernelEx(&cfg, k_attn_stream<true, false>, *tmQ, *tmK, *tmVt, *tmKs, *tmVs, a);
  return cudaLaunchKernelEx(&cfg, k_attn_stream<false, false>, *tmQ, *tmK, *tmVt, *tmKs, *tmVs, a);
}
