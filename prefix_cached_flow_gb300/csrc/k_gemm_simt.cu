// CUDA-core GEMMs and the W2A8 building blocks.
//
// * k_gemm_simt: out[z][t][n] = sum_{k in split z} X[t][k] W[n][k] in fp32
//   (fp32 config, the create-time time-conditioning table, and a diagnostic
//   path for bf16), or the K/V-cache scatter of the prefix projection
//   K_C = Z W_K, V_C = Z W_V ("vla.cpp: A Unified Inference Runtime for
//   Vision-Language-Action Models", §III-B Eq. (2)).
// * k_ternary_simt: exact integer sum_j a_tj q_nj with dp4a, where a are the
//   int8 activation codes and q the ternary weights decoded from four 2-bit
//   codes per byte (§III-D Eq. (4)).
// * k_quantize_rows / k_ternary_finish: Eq. (4) as standalone operations.
#include "vla_common.cuh"

namespace {

constexpr int BM = 64, BNS = 64, BK = 32;

template <typename TX, typename TW>
__global__ void __launch_bounds__(256) k_gemm_simt(const TX* __restrict__ X, int ldx, const TW* __restrict__ W,
                                                   int ldw, int T, int N, int K, int k_per_split,
                                                   float* __restrict__ out, size_t split_stride, int ldo,
                                                   KvScatter kv, int scatter) {
  __shared__ float Xs[BK][BM + 4];
  __shared__ float Ws[BK][BNS + 4];
  const int t0 = blockIdx.x * BM, n0 = blockIdx.y * BNS, z = blockIdx.z;
  const int kbeg = z * k_per_split;
  const int kend = min(K, kbeg + k_per_split);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    for (int idx = threadIdx.x; idx < BM * BK; idx += 256) {
      const int r = idx / BK, c = idx - r * BK;
      const int t = t0 + r, k = k0 + c;
      Xs[c][r] = (t < T && k < kend) ? to_f(X[(size_t)t * ldx + k]) : 0.f;
      const int n = n0 + r;
      Ws[c][r] = (n < N && k < kend) ? to_f(W[(size_t)n * ldw + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = Xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      if (!scatter) {
        out[(size_t)z * split_stride + (size_t)t * ldo + n] = acc[i][j];
      } else {
        // n -> (layer, K|V, kv head, dim); t -> (observation, prefix token)
        const int kvdim = kv.n_kv * kv.d_h;
        const int l = n / (2 * kvdim);
        const int rem = n - l * 2 * kvdim;
        const int which = rem / kvdim;
        const int r2 = rem - which * kvdim;
        const int g = r2 / kv.d_h, e = r2 - g * kv.d_h;
        const int b = t / kv.P, p = t - b * kv.P;
        if (which == 0)
          ((TW*)kv.kc)[((((size_t)l * kv.B + b) * kv.n_kv + g) * kv.P + p) * kv.d_h + e] = from_f<TW>(acc[i][j]);
        else
          ((TW*)kv.vc)[((((size_t)l * kv.B + b) * kv.n_kv + g) * kv.d_h + e) * kv.P8 + p] = from_f<TW>(acc[i][j]);
      }
    }
  }
}

// byte of four 2-bit codes -> four int8 ternary values (code - 1), little endian
__device__ __forceinline__ int decode_ternary_byte(uint32_t byte) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = (int)((byte >> (2 * i)) & 3u);
    w |= ((uint32_t)(c - 1) & 0xFFu) << (8 * i);
  }
  return (int)w;
}

constexpr int TBM = 64, TBN = 64, TBK = 64;  // TBK int8 per row = 16 words

__global__ void __launch_bounds__(256) k_ternary_simt(const int8_t* __restrict__ a, int lda,
                                                      const uint8_t* __restrict__ q, int T, int N, int K,
                                                      int k_per_split, float* __restrict__ out,
                                                      size_t split_stride, int ldo) {
  __shared__ int As[TBM][TBK / 4 + 1];
  __shared__ int Qs[TBN][TBK / 4 + 1];
  __shared__ int lut[256];
  for (int i = threadIdx.x; i < 256; i += 256) lut[i] = decode_ternary_byte((uint32_t)i);
  const int t0 = blockIdx.x * TBM, n0 = blockIdx.y * TBN, z = blockIdx.z;
  const int kbeg = z * k_per_split;
  const int kend = min(K, kbeg + k_per_split);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  int acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0;
  const int kq = K / 4;
  __syncthreads();
  for (int k0 = kbeg; k0 < kend; k0 += TBK) {
    for (int idx = threadIdx.x; idx < TBM * (TBK / 4); idx += 256) {
      const int r = idx / (TBK / 4), w = idx - r * (TBK / 4);
      const int t = t0 + r, kw = k0 / 4 + w;
      As[r][w] = (t < T && kw * 4 < kend) ? *(const int*)(a + (size_t)t * lda + kw * 4) : 0;
      const int n = n0 + r;
      Qs[r][w] = (n < N && kw * 4 < kend) ? lut[q[(size_t)n * kq + kw]] : 0;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < TBK / 4; ++w) {
      int av[4], qv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[ty * 4 + i][w];
#pragma unroll
      for (int j = 0; j < 4; ++j) qv[j] = Qs[tx * 4 + j][w];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __dp4a(av[i], qv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) out[(size_t)z * split_stride + (size_t)t * ldo + n] = (float)acc[i][j];
    }
  }
}

__global__ void k_quantize_rows(const float* __restrict__ x, int K, int8_t* __restrict__ a,
                                float* __restrict__ alpha) {
  extern __shared__ float sm[];
  float* row = sm;
  float* red = sm + K;
  const int m = blockIdx.x;
  for (int i = threadIdx.x; i < K; i += blockDim.x) row[i] = x[(size_t)m * K + i];
  __syncthreads();
  const float al = quantize_row_block(row, K, a + (size_t)m * K, nullptr, red);
  if (threadIdx.x == 0) alpha[m] = al;
}

__global__ void k_ternary_finish(const float* __restrict__ part, int M, int N, const float* __restrict__ alpha,
                                 float beta, uint16_t* __restrict__ y, int32_t* __restrict__ acc) {
  const size_t n_el = (size_t)M * N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_el; i += (size_t)gridDim.x * blockDim.x) {
    const int m = (int)(i / N);
    const float s = part[i];
    const float v = w2a8_scale(s, alpha[m], beta);
    y[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    if (acc) acc[i] = (int32_t)s;
  }
}

__global__ void k_check_codes(const uint8_t* __restrict__ q, size_t n, int* bad) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const uint32_t b = q[i];
    if ((b & 0x55u) & ((b >> 1) & 0x55u)) atomicOr(bad, 1);
  }
}

}  // namespace

cudaError_t launch_gemm_simt(int x_bf16, const void* X, int ldx, int w_bf16, const void* W, int ldw, int T, int N,
                             int K, int splits, float* out, size_t split_stride, int ldo, const KvScatter* kv,
                             cudaStream_t st) {
  if (splits < 1) splits = 1;
  int kps = (K + splits - 1) / splits;
  kps = (kps + BK - 1) / BK * BK;
  splits = (K + kps - 1) / kps;
  dim3 grid((T + BM - 1) / BM, (N + BNS - 1) / BNS, splits);
  KvScatter kvs = kv ? *kv : KvScatter{};
  const int sc = kv ? 1 : 0;
  if (!x_bf16 && !w_bf16)
    k_gemm_simt<float, float><<<grid, 256, 0, st>>>((const float*)X, ldx, (const float*)W, ldw, T, N, K, kps, out,
                                                    split_stride, ldo, kvs, sc);
  else if (!x_bf16 && w_bf16)
    k_gemm_simt<float, bf16><<<grid, 256, 0, st>>>((const float*)X, ldx, (const bf16*)W, ldw, T, N, K, kps, out,
                                                   split_stride, ldo, kvs, sc);
  else if (x_bf16 && w_bf16)
    k_gemm_simt<bf16, bf16><<<grid, 256, 0, st>>>((const bf16*)X, ldx, (const bf16*)W, ldw, T, N, K, kps, out,
                                                  split_stride, ldo, kvs, sc);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_ternary_simt(const int8_t* a, int lda, const uint8_t* q, int T, int N, int K, int splits,
                                float* out, size_t split_stride, int ldo, cudaStream_t st) {
  if (splits < 1) splits = 1;
  int kps = (K + splits - 1) / splits;
  kps = (kps + TBK - 1) / TBK * TBK;
  splits = (K + kps - 1) / kps;
  dim3 grid((T + TBM - 1) / TBM, (N + TBN - 1) / TBN, splits);
  k_ternary_simt<<<grid, 256, 0, st>>>(a, lda, q, T, N, K, kps, out, split_stride, ldo);
  return cudaGetLastError();
}

int simt_effective_splits(int K, int splits, int align) {
  if (splits < 1) splits = 1;
  int kps = (K + splits - 1) / splits;
  kps = (kps + align - 1) / align * align;
  return (K + kps - 1) / kps;
}

cudaError_t simt_kernels_init() {
  return set_max_dyn_smem(k_quantize_rows);
}

cudaError_t launch_quantize_rows(const float* x, int M, int K, int8_t* a, float* alpha, cudaStream_t st) {
  const size_t smem = (size_t)(K + 32) * sizeof(float);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  k_quantize_rows<<<M, 256, smem, st>>>(x, K, a, alpha);
  return cudaGetLastError();
}

cudaError_t launch_ternary_finish(const float* part, int M, int N, const float* alpha, float beta, uint16_t* y,
                                  int32_t* acc, cudaStream_t st) {
  const size_t n = (size_t)M * N;
  const int blocks = (int)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
  k_ternary_finish<<<blocks, 256, 0, st>>>(part, M, N, alpha, beta, y, acc);
  return cudaGetLastError();
}

cudaError_t launch_check_ternary_codes(const uint8_t* q, size_t nbytes, int* bad, cudaStream_t st) {
  const int blocks = (int)((nbytes + 255) / 256 < 8192 ? (nbytes + 255) / 256 : 8192);
  k_check_codes<<<blocks, 256, 0, st>>>(q, nbytes, bad);
  return cudaGetLastError();
}
