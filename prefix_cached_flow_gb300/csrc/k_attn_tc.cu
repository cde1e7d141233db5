// Joint non-causal GQA attention on tcgen05 ("vla.cpp: A Unified Inference
// Runtime for Vision-Language-Action Models", §III-B Eq. (2)):
//   o = softmax(Q [K_C ; K_s]^T / sqrt(d_h) + M) [V_C ; V_s],  M = 0,
// for the action queries of every head sharing one K/V head, over the cached
// prefix keys followed by the action tokens' own keys.
//
// A thread-block cluster of CS CTAs handles one 128-row query tile of one
// (observation, K/V head); rows are (query head within the group, action
// token).  Ranks 0..CS-2 each take KC consecutive prefix keys, rank CS-1 the
// action keys.  Per CTA:
//   S = Q K^T      tcgen05, A = Q [128][d_h], B = K chunk [KC][d_h]   -> TMEM
//   P = exp2(S log2e / sqrt(d_h) - m)   one thread per query row, bf16 into
//                                       a 128-byte-swizzled tile in smem
//   O = P V        tcgen05, A = P [128][KC], B = V^T chunk [d_h][KC] -> TMEM
// V is stored transposed so that both MMAs read K-major operands.  The ranks
// then merge: every rank publishes its unnormalised O in bf16 and each row's
// running maximum m_r and sum l_r through L2, one cluster barrier
// (release/acquire) makes them visible, and rank r weights the ranks' O by
// w_c = exp2(m_c - M) / sum_c' exp2(m_c' - M) l_c' (M the largest m over
// ranks with visible keys), sums a d_h/CS-column slice over the ranks in fp32
// (fixed order, deterministic) and writes bf16 o [B*H][n_q*d_h] (fp32 for the
// W2A8 quantiser).
// The prefix tiles are loaded before griddepcontrol.wait (they do not
// depend on the previous kernel); Q and the action keys/values after it.
#include "vla_common.cuh"

namespace {

struct AttnSmem {
  uint32_t q, k, v, p, bars, slot, ml;
  uint32_t total;
};

__host__ __device__ inline AttnSmem attn_layout(int d_h, int kc) {
  const int nsub = d_h / 64;
  const int ksub = (kc + 63) / 64;
  AttnSmem s;
  s.q = 0;                                           // nsub x [128][64] bf16
  s.k = s.q + nsub * 16384;                          // nsub x [kc][64]  (1024-aligned slices)
  const uint32_t kslice = ((uint32_t)kc * 128u + 1023u) & ~1023u;
  s.v = s.k + nsub * kslice;                         // ksub x [d_h][64]
  s.p = s.v + ksub * d_h * 128;                      // ksub x [128][64]
  const uint32_t end = s.p + ksub * 16384;
  s.bars = (end + 7u) & ~7u;                         // 3 mbarriers
  s.slot = s.bars + 3 * 8;
  s.ml = s.slot + 16;                                // [128] m, [128] l
  s.total = s.ml + 2 * 128 * 4;
  return s;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

template <bool O32, int CS, bool MASKED>
__global__ void __launch_bounds__(128, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ CUtensorMap tmKs,
              const __grid_constant__ CUtensorMap tmVs, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int dh = a.d_h;  // cluster size CS is a template parameter (code size: only CS ranks' exchanges)
  const int nsub = dh / 64;
  const bool suffix = (int)blockIdx.x == CS - 1;
  const int kc = suffix ? a.kc_s : a.kc;             // keys this rank's tiles hold
  const int ksub = (kc + 63) / 64;
  const AttnSmem L = attn_layout(dh, a.kc > a.kc_s ? a.kc : a.kc_s);
  const uint32_t kslice = ((uint32_t)kc * 128u + 1023u) & ~1023u;
  uint8_t* Qs = smem + L.q;
  uint8_t* Ks = smem + L.k;
  uint8_t* Vt = smem + L.v;
  uint8_t* Ps = smem + L.p;
  uint64_t* bars = (uint64_t*)(smem + L.bars);  // 0: K/V, 1: Q, 2: MMA done
  uint32_t* tmem_slot = (uint32_t*)(smem + L.slot);
  float* sm_m = (float*)(smem + L.ml);
  float* sm_l = sm_m + 128;
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x, qt = blockIdx.y, bg = blockIdx.z;
  const int b = bg / a.n_kv, gk = bg - b * a.n_kv;
  const int key0 = suffix ? 0 : rank * a.kc;
  const int avail = (suffix ? (a.no_suffix ? 0 : a.H) : a.P) - key0;  // cross layers: no action keys
  const int nk = avail < 0 ? 0 : (avail < kc ? avail : kc);
  uint32_t ncols = 32;
  while (ncols < (uint32_t)dh || ncols < (uint32_t)kc) ncols <<= 1;
  const uint32_t kv_bytes = (uint32_t)nsub * (uint32_t)kc * 128u + (uint32_t)ksub * (uint32_t)dh * 128u;
  const uint32_t q_bytes = (uint32_t)nsub * 16384u;
  VLA_TL(a.tl, 0, 0);

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
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

  // Prefix K / V^T tiles: cache data, independent of the previous kernel.
  if (threadIdx.x == 0 && !suffix && nk > 0) {
    const int z = (a.layer * a.B + b) * a.n_kv + gk;
    mbar_arrive_expect_tx(&bars[0], kv_bytes);
    for (int s = 0; s < nsub; ++s) tma_load_3d(Ks + (size_t)s * kslice, &tmK, &bars[0], s * 64, key0, z);
    for (int s = 0; s < ksub; ++s) tma_load_3d(Vt + (size_t)s * dh * 128, &tmVt, &bars[0], key0 + s * 64, 0, z);
  }
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  VLA_TL(a.tl, 0, 1);
  if (threadIdx.x == 0 && nk > 0) {
    if (suffix) {
      const int z = b * a.n_kv + gk;
      mbar_arrive_expect_tx(&bars[0], kv_bytes);
      for (int s = 0; s < nsub; ++s) tma_load_3d(Ks + (size_t)s * kslice, &tmKs, &bars[0], s * 64, 0, z);
      for (int s = 0; s < ksub; ++s) tma_load_3d(Vt + (size_t)s * dh * 128, &tmVs, &bars[0], s * 64, 0, z);
    }
    const int qrow = (b * a.n_q + gk * a.group) * a.H + qt * 128;
    mbar_arrive_expect_tx(&bars[1], q_bytes);
    for (int s = 0; s < nsub; ++s) tma_load_2d(Qs + (size_t)s * 16384, &tmQ, &bars[1], s * 64, qrow);
  }

  // S = Q K^T
  const uint32_t parity0 = 0;
  if (nk > 0) {
    if (warp == 1 && lane == 0) {
      const bool okw = mbar_wait(&bars[1], 0, a.status) && mbar_wait(&bars[0], 0, a.status);
      if (!okw) s_fail = 1;
      VLA_TL(a.tl, 32, 2);
      if (okw) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, kc);
        for (int s = 0; s < nsub; ++s) {
          const uint32_t qa = smem_u32(Qs + (size_t)s * 16384), ka = smem_u32(Ks + (size_t)s * kslice);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(tmem, sdesc_k128(qa + k * 32), sdesc_k128(ka + k * 32), idesc, (s > 0 || k > 0) ? 1u : 0u);
        }
      }
      umma_commit(&bars[2]);
    }
    __syncwarp();
    if (!mbar_wait(&bars[2], parity0, a.status)) s_fail = 1;
    tc_fence_after();
  }
  __syncthreads();
  const bool ok = s_fail == 0;
  VLA_TL(a.tl, 0, 3);

  // Softmax over this rank's keys, one query row per thread (two passes over TMEM).
  const int row = warp * 32 + lane;
  const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
  float m = -INFINITY, l = 0.f;
  const uint32_t* mrow = (!MASKED || suffix) ? nullptr : a.pmask + (size_t)b * a.pmw;
  if (ok && nk > 0) {
    // Two passes over TMEM in 32-column pieces.  Every CTA runs this code
    // once, so it is kept compact (rolled loops whose bodies repeat, instead
    // of holding the row in registers with fully unrolled code).  Columns in
    // [nk, 32-roundup of kc) are masked by a select; they lie inside the
    // TMEM allocation (at least 64 columns, d_h >= 64).
    float mxv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
    for (int c0 = 0; c0 < kc; c0 += 32) {
      uint32_t r[32];
      tmem_ld16_nowait(taddr + (uint32_t)c0, r);
      tmem_ld16_nowait(taddr + (uint32_t)(c0 + 16), r + 16);
      tmem_wait16(r);
      tmem_wait16(r + 16);
      const uint32_t mb = MASKED ? prefix_mask_window(mrow, a.pmw, key0 + c0) : 0xFFFFFFFFu;
      if (c0 + 32 <= nk && mb == 0xFFFFFFFFu) {  // a full visible piece (uniform over the CTA): no masks
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          float& mm = mxv[(u >> 1) & 3];
          asm("max.f32 %0, %0, %1, %2;" : "+f"(mm) : "f"(__uint_as_float(r[u])), "f"(__uint_as_float(r[u + 1])));
        }
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u)
          mxv[u & 3] = fmaxf(mxv[u & 3], (c0 + u < nk && ((mb >> u) & 1u)) ? __uint_as_float(r[u]) : -INFINITY);
      }
    }
    m = fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])) * a.scale_log2;  // the scale is positive
    VLA_TL(a.tl, 0, 11);
    const float nm = -m;
    float lv[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t pa = smem_u32(Ps);
#pragma unroll 1
    for (int c0 = 0; c0 < kc; c0 += 32) {
      uint32_t r[32];
      tmem_ld16_nowait(taddr + (uint32_t)c0, r);
      tmem_ld16_nowait(taddr + (uint32_t)(c0 + 16), r + 16);
      tmem_wait16(r);
      tmem_wait16(r + 16);
      const uint32_t mb = MASKED ? prefix_mask_window(mrow, a.pmw, key0 + c0) : 0xFFFFFFFFu;
      const bool masked = c0 + 32 > nk || mb != 0xFFFFFFFFu;  // the last, partial piece or hidden keys
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 8-key chunks
        float p[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = c0 + q * 8 + u;
          p[u] = fast_exp2(fmaf(__uint_as_float(r[q * 8 + u]), a.scale_log2, nm));
          if (masked) p[u] = (j < nk && ((mb >> (q * 8 + u)) & 1u)) ? p[u] : 0.f;
          lv[u & 3] += p[u];
        }
        uint4 pk;
        pk.x = pack_bf16x2(p[0], p[1]);
        pk.y = pack_bf16x2(p[2], p[3]);
        pk.z = pack_bf16x2(p[4], p[5]);
        pk.w = pack_bf16x2(p[6], p[7]);
        const int ch = c0 / 8 + q;  // 8-key chunk index within the rank's keys
        if (ch * 8 < kc)
          st_shared_v4_u32(pa + (uint32_t)(ch >> 3) * 16384u + sw128_offset((uint32_t)row, (uint32_t)(ch & 7)), pk);
      }
    }
    l = (lv[0] + lv[1]) + (lv[2] + lv[3]);
  }
  VLA_TL(a.tl, 0, 8);
  sm_m[row] = m;
  sm_l[row] = l;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // O = P V (overwrites S's TMEM columns: every S read has completed).
  if (nk > 0) {
    if (warp == 1 && lane == 0) {
      if (ok) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, dh);
        const uint32_t pa = smem_u32(Ps), va = smem_u32(Vt);
        for (int kk = 0; kk < kc / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u;
          const uint32_t voff = (uint32_t)(kk >> 2) * (uint32_t)dh * 128u + (uint32_t)(kk & 3) * 32u;
          umma_bf16(tmem, sdesc_k128(pa + off), sdesc_k128(va + voff), idesc, kk > 0 ? 1u : 0u);
        }
      }
      umma_commit(&bars[2]);
    }
    __syncwarp();
    if (!mbar_wait(&bars[2], parity0 ^ 1u, a.status)) s_fail = 1;
    tc_fence_after();
  }
  VLA_TL(a.tl, 0, 9);

  // Publish this rank's unnormalised O (bf16) and each row's (m, l) through
  // L2; O is interleaved as [d_h/8][128 rows][8] so that a warp's 32 rows
  // form one 512-byte run.  One cluster barrier (release/acquire) then makes
  // every rank's part visible to the merge.
  const int nrows = (a.group * a.H - qt * 128) < 128 ? (a.group * a.H - qt * 128) : 128;
  const size_t cl = (size_t)bg * a.n_qt + qt;  // this cluster's query tile
  if (s_fail == 0 && nk > 0) {
    uint4* dst = (uint4*)(a.xo + (cl * CS + rank) * 128 * (size_t)dh) + row;
    for (int c0 = 0; c0 < dh; c0 += 64) {  // 64 columns per TMEM wait
      uint32_t r[64];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld16_nowait(taddr + (uint32_t)(c0 + q * 16), r + q * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_wait16(r + q * 16);
      if (row < nrows) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t* w = r + q * 8;
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1]));
          u.y = pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3]));
          u.z = pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5]));
          u.w = pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7]));
          __stcg(dst + (size_t)(c0 / 8 + q) * 128, u);
        }
      }
    }
    if (row < nrows) __stcg(&a.xml[(cl * CS + rank) * 128 + row], make_float2(m, l));
  }
  cluster_sync_all();
  VLA_TL(a.tl, 0, 5);

  // Rank r sums columns [r*dh/CS, (r+1)*dh/CS) over the ranks that held keys
  // (fixed order, fp32) and writes o: one query row per thread.
  const int cols = dh / CS;
  const int q8 = cols / 8;  // 8-column groups in this slice
  if (s_fail == 0 && row < nrows) {
    // ranks that held keys: the prefix ranks with keys, the action-key rank
    // unless this is a cross-attention layer
    auto held_rank = [&](int c) { return c == CS - 1 ? a.no_suffix == 0 : c * a.kc < a.P; };
    // merge weights of this row: w_c = 2^(m_c - M) / sum_c 2^(m_c - M) l_c,
    // M = max_c m_c over the ranks with visible keys (a rank whose keys are
    // all hidden has l_c = 0 and weight 0)
    float mrow[CS], lrow[CS], wgt[CS];
#pragma unroll
    for (int c = 0; c < CS; ++c) {
      const float2 ml = held_rank(c) ? __ldcg(&a.xml[(cl * CS + c) * 128 + row]) : make_float2(-INFINITY, 0.f);
      mrow[c] = ml.x;
      lrow[c] = ml.y;
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < CS; ++c)
      if (lrow[c] > 0.f) M = fmaxf(M, mrow[c]);
    float den = 0.f;
#pragma unroll
    for (int c = 0; c < CS; ++c) {
      wgt[c] = lrow[c] > 0.f ? fast_exp2(mrow[c] - M) : 0.f;
      den += wgt[c] * lrow[c];
    }
    const float inv = 1.f / den;
#pragma unroll
    for (int c = 0; c < CS; ++c) wgt[c] *= inv;
    const int rg = qt * 128 + row;  // row within the group: (head, token)
    const int jj = rg / a.H, i = rg - jj * a.H;
    const int j = gk * a.group + jj;
    bf16* out = a.o + ((size_t)b * a.H + i) * (size_t)(a.n_q * dh) + (size_t)j * dh + rank * cols;
    for (int c8 = 0; c8 < q8; c8 += 2) {
      uint4 v[2][CS];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < CS; ++c) {
          const bool held = (c8 + h) < q8 && held_rank(c);
          v[h][c] = held ? __ldcg((const uint4*)(a.xo + (cl * CS + c) * 128 * (size_t)dh) +
                                  (size_t)(rank * q8 + c8 + h) * 128 + row)
                         : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (c8 + h >= q8) break;
        float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < CS; ++c) {
          const uint32_t w[4] = {v[h][c].x, v[h][c].y, v[h][c].z, v[h][c].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            sum[2 * u] = fmaf(wgt[c], __uint_as_float(w[u] << 16), sum[2 * u]);
            sum[2 * u + 1] = fmaf(wgt[c], __uint_as_float(w[u] & 0xFFFF0000u), sum[2 * u + 1]);
          }
        }
        if (O32) {
          float4* o32 = (float4*)(a.o32 + ((size_t)b * a.H + i) * (size_t)(a.n_q * dh) + (size_t)j * dh + rank * cols +
                                  (c8 + h) * 8);
          o32[0] = make_float4(sum[0], sum[1], sum[2], sum[3]);
          o32[1] = make_float4(sum[4], sum[5], sum[6], sum[7]);
        } else {
          uint4 o4;
          o4.x = pack_bf16x2(sum[0], sum[1]); o4.y = pack_bf16x2(sum[2], sum[3]);
          o4.z = pack_bf16x2(sum[4], sum[5]); o4.w = pack_bf16x2(sum[6], sum[7]);
          *(uint4*)(out + (c8 + h) * 8) = o4;
        }
      }
    }
  }
  VLA_TL(a.tl, 0, 6);

  // Drain the TMA copies (complete unless a wait timed out) and free TMEM.
  if (threadIdx.x == 0 && nk > 0) {
    mbar_drain(&bars[0], 0);
    mbar_drain(&bars[1], 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

}  // namespace

size_t attn_tc_smem_bytes(int d_h, int kc) { return 1024 + attn_layout(d_h, kc).total; }

template <bool O32, int CS>
cudaError_t attn_init_one() {
  cudaError_t e = set_max_dyn_smem(k_attn_tc<O32, CS, false>);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_attn_tc<O32, CS, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) e = set_max_dyn_smem(k_attn_tc<O32, CS, true>);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_attn_tc<O32, CS, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t attn_kernels_init() {
  cudaError_t e = attn_init_one<false, 8>();
  if (e == cudaSuccess) e = attn_init_one<false, 16>();
  if (e == cudaSuccess) e = attn_init_one<true, 8>();
  if (e == cudaSuccess) e = attn_init_one<true, 16>();
  return e;
}

cudaError_t launch_attn_tc(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmVt,
                           const CUtensorMap* tmKs, const CUtensorMap* tmVs, const AttnArgs& a, cudaStream_t st) {
  if (a.d_h % 64 || a.d_h > 256 || a.d_h < 64 || (a.cs != 8 && a.cs != 16) || a.kc < 16 ||
      a.kc > 128 || a.kc % 16 || a.kc_s < 16 || a.kc_s > 128 || a.kc_s % 16 || (a.d_h / a.cs) % 8 || !a.xo ||
      !a.xml)
    return cudaErrorInvalidValue;
  const int kmax = a.kc > a.kc_s ? a.kc : a.kc_s;
  const size_t smem = attn_tc_smem_bytes(a.d_h, kmax);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.cs, a.n_qt, a.B * a.n_kv);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
#define VLA_ATTN_GO(O, C, M) return cudaLaunchKernelEx(&cfg, k_attn_tc<O, C, M>, *tmQ, *tmK, *tmVt, *tmKs, *tmVs, a)
  const bool m = a.pmask != nullptr;  // the masked instantiations only when a mask is given
  if (a.cs == 8) {
    if (a.o32) { if (m) VLA_ATTN_GO(true, 8, true); VLA_ATTN_GO(true, 8, false); }
    if (m) VLA_ATTN_GO(false, 8, true);
    VLA_ATTN_GO(false, 8, false);
  }
  if (a.o32) { if (m) VLA_ATTN_GO(true, 16, true); VLA_ATTN_GO(true, 16, false); }
  if (m) VLA_ATTN_GO(false, 16, true);
  VLA_ATTN_GO(false, 16, false);
#undef VLA_ATTN_GO
}
