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
// Warp roles (192 threads):
//   warps 0-3  softmax and epilogue, one query row per thread (TMEM lane)
//   warp 4     TMA producer: Q once, K_j and V_j^T into a two-stage ring
//   warp 5     MMA issuer:   S_j = Q K_j^T into one of two TMEM S buffers,
//                            O += P_j V_j into the TMEM O accumulator
// Per chunk j the softmax thread reads its row of S_j, updates the running
// maximum m, writes P_j = exp2(S_j log2e / sqrt(d_h) - m) in bf16 to shared
// memory and adds it to the row sum l.  m is raised lazily: only when a chunk
// maximum exceeds it by more than 2^8 in the exponent are O (in TMEM) and l
// rescaled, so P never exceeds 256 and the final o = O / l is unchanged in
// exact arithmetic.  S_{j+1} runs on the tensor cores while P_j is computed;
// P_j V_j runs while S_{j+1} is read.
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
  s.slot = s.bars + 16 * 8;
  s.total = s.slot + 16;
  return s;
}

enum { B_Q = 0, B_KVF = 1, B_KVE = 3, B_SF = 5, B_PF = 7, B_PV = 9, B_FIN = 11, N_BARS = 12 };

__device__ __forceinline__ void tma_load_3d_s(void* dst, const void* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

template <bool O32>
__global__ void __launch_bounds__(192, 1)
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
  const uint32_t ncols = dh + 2 * KB <= 256 ? 256u : 512u;  // O (d_h columns) + two S buffers
  const uint32_t s_col = (uint32_t)dh;

  if (threadIdx.x == 0) {
    s_fail = 0;
    mbar_init(&bars[B_Q], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_KVF + i], 1);
      mbar_init(&bars[B_KVE + i], 1);
      mbar_init(&bars[B_SF + i], 1);
      mbar_init(&bars[B_PF + i], 128);
      mbar_init(&bars[B_PV + i], 1);
    }
    mbar_init(&bars[B_FIN], 1);
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

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int zc = (a.layer * a.B + b) * a.n_kv + gk;
      const int zs = b * a.n_kv + gk;
      const uint32_t kv_bytes = (uint32_t)nsub * 8192u + (uint32_t)dh * 128u;
      auto issue = [&](int j) {
        const int st = j & 1;
        uint8_t* kd = Ks + (size_t)st * nsub * 8192;
        uint8_t* vd = Vs + (size_t)st * dh * 128;
        mbar_arrive_expect_tx(&bars[B_KVF + st], kv_bytes);
        if (j < n_pre) {
          for (int s = 0; s < nsub; ++s) tma_load_3d_s(kd + (size_t)s * 8192, &tmK, &bars[B_KVF + st], s * 64, j * KB, zc);
          tma_load_3d_s(vd, &tmVt, &bars[B_KVF + st], j * KB, 0, zc);
        } else {
          const int k0 = (j - n_pre) * KB;
          for (int s = 0; s < nsub; ++s) tma_load_3d_s(kd + (size_t)s * 8192, &tmKs, &bars[B_KVF + st], s * 64, k0, zs);
          tma_load_3d_s(vd, &tmVs, &bars[B_KVF + st], k0, 0, zs);
        }
      };
      // The cached prefix does not depend on the previous kernel: its first
      // two chunks are in flight before the grid dependency wait.
      int j = 0;
      for (; j < 2 && j < n_pre; ++j) issue(j);
      griddep_wait();
      mbar_arrive_expect_tx(&bars[B_Q], (uint32_t)nsub * 16384u);
      const int qrow = (b * a.n_q + gk * a.group) * a.H + qt * 128;
      for (int s = 0; s < nsub; ++s) tma_load_2d(Qs + (size_t)s * 16384, &tmQ, &bars[B_Q], s * 64, qrow);
      for (; j < nch; ++j) {
        if (j >= 2 && !mbar_wait(&bars[B_KVE + (j & 1)], (uint32_t)((j - 2) >> 1) & 1u, a.status)) {
          s_fail = 1;
          break;
        }
        issue(j);
      }
      // Own copies land before the CTA can exit (normally already consumed).
      const int issued = j;
      for (int i = issued - 2 < 0 ? 0 : issued - 2; i < issued; ++i)
        mbar_drain(&bars[B_KVF + (i & 1)], (uint32_t)(i >> 1) & 1u);
      mbar_drain(&bars[B_Q], 0);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    griddep_wait();
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, KB);
      const uint32_t idesc_o = idesc_bf16_f32(128, dh);
      bool ok = mbar_wait(&bars[B_Q], 0, a.status);
      auto pv = [&](int i) -> bool {
        const int st = i & 1;
        if (!mbar_wait(&bars[B_PF + st], (uint32_t)(i >> 1) & 1u, a.status)) return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(Ps + (size_t)st * 16384), va = smem_u32(Vs + (size_t)st * dh * 128);
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk)
          umma_bf16(tmem, sdesc_k128(pa + kk * 32), sdesc_k128(va + kk * 32), idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars[B_PV + st]);
        umma_commit(&bars[B_KVE + st]);
        return true;
      };
      int j = 0;
      for (; ok && j < nch; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&bars[B_KVF + st], (uint32_t)(j >> 1) & 1u, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ka = smem_u32(Ks + (size_t)st * nsub * 8192);
        for (int s = 0; s < nsub; ++s) {
          const uint32_t qa = smem_u32(Qs + (size_t)s * 16384), kb = ka + (uint32_t)s * 8192u;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(tmem + s_col + (uint32_t)(st * KB), sdesc_k128(qa + k * 32), sdesc_k128(kb + k * 32), idesc_s,
                      (s > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_SF + st]);
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
    // ---------------- softmax + epilogue (warps 0-3) ----------------
    griddep_wait();
    const int row = threadIdx.x;  // query row in the tile = TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nch; ++j) {
      const int st = j & 1;
      if (!__all_sync(~0u, mbar_wait(&bars[B_SF + st], (uint32_t)(j >> 1) & 1u, a.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int nk = j < n_pre ? (a.P - j * KB < KB ? a.P - j * KB : KB)
                               : (a.H - (j - n_pre) * KB < KB ? a.H - (j - n_pre) * KB : KB);
      uint32_t sr[KB];
#pragma unroll
      for (int q = 0; q < KB / 16; ++q) tmem_ld16_nowait(trow + s_col + (uint32_t)(st * KB + q * 16), sr + q * 16);
#pragma unroll
      for (int q = 0; q < KB / 16; ++q) tmem_wait16(sr + q * 16);
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < KB; ++u)
        if (u < nk) mx = fmaxf(mx, __uint_as_float(sr[u]) * a.scale_log2);
      // The decision is per warp (tcgen05.ld / st are warp-collective); a
      // lane whose own maximum did not grow scales by 1.
      if (__any_sync(~0u, mx > m_used + RESCALE_LOG2)) {
        const float m_new = fmaxf(m_used, mx);
        if (j > 0) {
          // O holds sum_{i<j} P_i V_i at the old maximum: wait for the last
          // product, then scale the row by 2^(m_used - m_new) in place.
          if (!__all_sync(~0u, mbar_wait(&bars[B_PV + ((j - 1) & 1)], (uint32_t)((j - 1) >> 1) & 1u, a.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = fast_exp2(m_used - m_new);
          for (int c0 = 0; c0 < dh; c0 += 64) {
            uint32_t r[64];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16_nowait(trow + (uint32_t)(c0 + q * 16), r + q * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_wait16(r + q * 16);
#pragma unroll
            for (int u = 0; u < 64; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * f);
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_st16(trow + (uint32_t)(c0 + q * 16), r + q * 16);
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
#pragma unroll
      for (int q = 0; q < KB / 8; ++q) {
        float p[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = q * 8 + u;
          p[u] = c < nk ? fast_exp2(__uint_as_float(sr[c]) * a.scale_log2 - m_used) : 0.f;
          l += p[u];
        }
        uint4 pk;
        pk.x = pack_bf16x2(p[0], p[1]);
        pk.y = pack_bf16x2(p[2], p[3]);
        pk.z = pack_bf16x2(p[4], p[5]);
        pk.w = pack_bf16x2(p[6], p[7]);
        st_shared_v4_u32(pa + sw128_offset((uint32_t)row, (uint32_t)q), pk);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[B_PF + st]);
    }
    if (!ok) s_fail = 1;
    // Epilogue: o = O / l for the valid rows of the tile.
    if (ok && __all_sync(~0u, mbar_wait(&bars[B_PV + ((nch - 1) & 1)], (uint32_t)((nch - 1) >> 1) & 1u, a.status))) {
      tc_fence_after();
      const int nrows = (a.group * a.H - qt * 128) < 128 ? (a.group * a.H - qt * 128) : 128;
      const float inv = 1.f / l;
      const int rg = qt * 128 + row;  // (query head within the group, action token)
      const int jj = rg / a.H, i = rg - jj * a.H;
      const size_t obase = ((size_t)b * a.H + i) * (size_t)(a.n_q * dh) + (size_t)(gk * a.group + jj) * dh;
      for (int c0 = 0; c0 < dh; c0 += 64) {
        uint32_t r[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16_nowait(trow + (uint32_t)(c0 + q * 16), r + q * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_wait16(r + q * 16);
        if (row < nrows) {
          if (O32) {
            float4* dst = (float4*)(a.o32 + obase + c0);
#pragma unroll
            for (int q = 0; q < 16; ++q)
              dst[q] = make_float4(__uint_as_float(r[4 * q]) * inv, __uint_as_float(r[4 * q + 1]) * inv,
                                   __uint_as_float(r[4 * q + 2]) * inv, __uint_as_float(r[4 * q + 3]) * inv);
          } else {
            uint4* dst = (uint4*)(a.o + obase + c0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t* w = r + q * 8;
              uint4 u;
              u.x = pack_bf16x2(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv);
              u.y = pack_bf16x2(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv);
              u.z = pack_bf16x2(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv);
              u.w = pack_bf16x2(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv);
              dst[q] = u;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
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
  if (a.d_h % 64 || a.d_h > 256 || a.d_h < 64 || a.P < 1 || a.H < 1 || a.n_qt < 1 ||
      a.n_qt * 128 < a.group * a.H)
    return cudaErrorInvalidValue;
  const size_t smem = attn_stream_smem_bytes(a.d_h);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_qt, a.B * a.n_kv, 1);
  cfg.blockDim = dim3(192, 1, 1);
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
