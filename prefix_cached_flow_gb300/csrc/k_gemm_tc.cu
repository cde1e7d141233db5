// tcgen05 GEMM for sm_103a: bf16 operands staged by TMA into 128-byte
// swizzled shared-memory tiles, fp32 accumulators in TMEM.
//
// D[n][t] = sum_k W[n][k] X[t][k]: the weight rows are the MMA's M = 128
// operand (A) and the action / prefix tokens the N operand (B, 16..256 rows),
// so a batch-1 step with a few dozen tokens still streams its weights as
// full 128-row tiles ("swap-AB").  Used for the prefix projection
// K_C = Z W_K, V_C = Z W_V ("vla.cpp: A Unified Inference Runtime for
// Vision-Language-Action Models", §III-B Eq. (2)) with a K/V-cache scatter
// epilogue, and for the expert's linear maps with fp32 split-K partials.
//
// One CTA = 4 warps: warp 0 lane 0 issues TMA loads into a ring of `stages`
// buffers, warp 1 lane 0 issues the MMAs and releases each buffer with
// tcgen05.commit, then all four warps read the accumulator rows out of TMEM
// (warp w owns TMEM lanes 32w..32w+31).  Every wait is bounded.
#include "vla_common.cuh"

namespace {

constexpr uint32_t kABytes = 128 * 128;  // 128 weight rows x 64 bf16

__global__ void __launch_bounds__(128, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcGemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int BN = g.BN, NS = g.stages;
  const uint32_t b_bytes = (uint32_t)BN * 128u;
  const uint32_t stage_bytes = kABytes + b_bytes;
  uint64_t* full = (uint64_t*)(smem + (size_t)NS * stage_bytes);
  uint64_t* empty = full + NS;
  uint64_t* done = empty + NS;
  uint32_t* tmem_slot = (uint32_t*)(done + 1);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128;
  const int t0 = blockIdx.y * BN;
  const int kb0 = blockIdx.z * g.kb_per_split;
  const int nkb = min(g.kb_per_split, g.num_kb - kb0);
  uint32_t ncols = 32;
  while (ncols < (uint32_t)BN) ncols <<= 1;

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued = 0;
  if (warp == 0 && lane == 0) {
    // TMA producer: weights are read once per launch -> evict-first.
    const uint64_t pol_w = l2_policy_evict_first();
    for (int i = 0; i < nkb; ++i) {
      const int s = i % NS;
      if (i >= NS && !mbar_wait(&empty[s], ((i / NS) & 1) ^ 1, g.status)) {
        s_fail = 1;
        break;
      }
      uint8_t* sa = smem + (size_t)s * stage_bytes;
      mbar_arrive_expect_tx(&full[s], stage_bytes);
      tma_load_2d_hint(sa, &tmA, &full[s], (kb0 + i) * 64, g.a_row0 + m0, pol_w);
      tma_load_2d(sa + kABytes, &tmB, &full[s], (kb0 + i) * 64, t0);
      issued = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: 4 x (K = 16) per 64-wide k-block.
    const uint32_t idesc = idesc_bf16_f32(128, BN);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % NS;
      if (!mbar_wait(&full[s], (i / NS) & 1, g.status)) {
        s_fail = 1;
        break;
      }
      tc_fence_after();
      const uint32_t a_addr = smem_u32(smem + (size_t)s * stage_bytes);
      const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_bf16(tmem, sdesc_k128(a_addr + k * 32), sdesc_k128(b_addr + k * 32), idesc,
                  (i > 0 || k > 0) ? 1u : 0u);
      umma_commit(&empty[s]);
    }
    umma_commit(done);
  }
  __syncwarp();

  // Epilogue: TMEM -> registers -> global.
  if (!mbar_wait(done, 0, g.status)) s_fail = 1;
  tc_fence_after();
  __syncthreads();
  const bool ok = (s_fail == 0);
  const int row = warp * 32 + lane;
  const int n = m0 + row;
  const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
  if (ok) {
    for (int c0 = 0; c0 < BN; c0 += 16) {
      float v[16];
      tmem_ld16(taddr + (uint32_t)c0, v);
      if (n >= g.N) continue;
      if (g.mode == 0) {
        float* o = g.out + (size_t)blockIdx.z * g.split_stride + n;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = t0 + c0 + j;
          if (t < g.T) o[(size_t)t * g.ldo] = v[j];
        }
      } else {
        const KvScatter& kv = g.kv;
        const int kvdim = kv.n_kv * kv.d_h;
        const int l = n / (2 * kvdim);
        const int rem = n - l * 2 * kvdim;
        const int which = rem / kvdim;
        const int r2 = rem - which * kvdim;
        const int gg = r2 / kv.d_h, e = r2 - gg * kv.d_h;
        if (which == 0) {
          bf16* dst = (bf16*)kv.kc;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = t0 + c0 + j;
            if (t >= g.T) continue;
            const int b = t / kv.P, p = t - b * kv.P;
            dst[((((size_t)l * kv.B + b) * kv.n_kv + gg) * kv.P + p) * kv.d_h + e] = __float2bfloat16_rn(v[j]);
          }
        } else {
          // V_C^T: this thread's row (feature e) gets 16 consecutive tokens.
          bf16* dst = (bf16*)kv.vc;
          const int tb = t0 + c0;
          const int b0 = tb / kv.P, p0 = tb - b0 * kv.P;
          bf16* rowp = dst + ((((size_t)l * kv.B + b0) * kv.n_kv + gg) * kv.d_h + e) * kv.P8;
          if (tb + 15 < g.T && p0 + 15 < kv.P && (p0 & 7) == 0) {
            uint4 a, bq;
            a.x = pack_bf16x2(v[0], v[1]); a.y = pack_bf16x2(v[2], v[3]);
            a.z = pack_bf16x2(v[4], v[5]); a.w = pack_bf16x2(v[6], v[7]);
            bq.x = pack_bf16x2(v[8], v[9]); bq.y = pack_bf16x2(v[10], v[11]);
            bq.z = pack_bf16x2(v[12], v[13]); bq.w = pack_bf16x2(v[14], v[15]);
            *(uint4*)(rowp + p0) = a;
            *(uint4*)(rowp + p0 + 8) = bq;
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = tb + j;
              if (t >= g.T) continue;
              const int b = t / kv.P, p = t - b * kv.P;
              dst[((((size_t)l * kv.B + b) * kv.n_kv + gg) * kv.d_h + e) * kv.P8 + p] = __float2bfloat16_rn(v[j]);
            }
          }
        }
      }
    }
  }

  // Drain: make sure no TMA write into this CTA's shared memory is in flight.
  if (warp == 0 && lane == 0) {
    const int first = issued > NS ? issued - NS : 0;
    for (int i = first; i < issued; ++i) mbar_drain(&full[i % NS], (i / NS) & 1);
    mbar_drain(done, 0);  // the MMA warp always commits `done`
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiled_t get_encode() {
  static PFN_encodeTiled_t fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_encodeTiled_t)p;
  }
  return fn;
}

}  // namespace

int tc_encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows) {
  PFN_encodeTiled_t fn = get_encode();
  if (!fn) return -1;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)r;
}

cudaError_t tc_kernels_init() {
  return set_max_dyn_smem(k_gemm_tc);
}

int tc_encode_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                     uint32_t box_rows) {
  PFN_encodeTiled_t fn = get_encode();
  if (!fn) return -1;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)r;
}

int tc_encode_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows) {
  PFN_encodeTiled_t fn = get_encode();
  if (!fn) return -1;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)r;
}

int tc_encode_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                      uint64_t stride2_bytes, uint32_t box0, uint32_t box1) {
  PFN_encodeTiled_t fn = get_encode();
  if (!fn) return -1;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)r;
}

size_t tc_smem_bytes(int BN, int stages) {
  return (size_t)stages * (kABytes + (size_t)BN * 128) + 1024 /*alignment slack*/ + (2 * stages + 1) * 8 + 16;
}

cudaError_t launch_gemm_tc(const CUtensorMap* tmA, const CUtensorMap* tmB, const TcGemmArgs& a, int tiles_n,
                           int tiles_t, int splits, cudaStream_t st) {
  if (a.BN < 16 || a.BN > 256 || (a.BN % 16) != 0 || a.stages < 1) return cudaErrorInvalidValue;
  const size_t smem = tc_smem_bytes(a.BN, a.stages);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  dim3 grid(tiles_n, tiles_t, splits);
  k_gemm_tc<<<grid, 128, smem, st>>>(*tmA, *tmB, a);
  return cudaGetLastError();
}
