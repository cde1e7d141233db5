// Internal declarations shared by the libvla translation units.
//
// Device-side building blocks: hand-written inline PTX for sm_103a (mbarrier,
// TMA bulk tensor copies, tcgen05 MMA / TMEM), bounded waits that latch an
// error word instead of spinning forever, block reductions, and the Eq. (4)
// row quantiser ("vla.cpp: A Unified Inference Runtime for
// Vision-Language-Action Models", §III-D) that every W2A8 producer shares.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/vla.h"

typedef __nv_bfloat16 bf16;

// Device error word values (the first error is latched).
#define VLA_DEV_OK 0
#define VLA_DEV_TIMEOUT 6
#define VLA_DEV_ABORTED 7

// A bounded wait gives up after this long (ns of %globaltimer).
#define VLA_WAIT_LIMIT_NS 2000000000ull

// ---------------------------------------------------------------------------
// Scalar conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// Error latch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void latch_error(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Optional event trace (built only with -DVLA_TIMELINE): thread `who` of each
// CTA stores a timestamp for event `ev` (< 16) into tl[cta * 16 + ev]:
// %globaltimer (comparable across SMs and kernels, coarse), or with
// -DVLA_TIMELINE_CYCLES the SM's cycle counter (fine, comparable only within
// one CTA).
#ifdef VLA_TIMELINE_CYCLES
#define VLA_TL_NOW() ((unsigned long long)clock64())
#else
#define VLA_TL_NOW() globaltimer_ns()
#endif
#ifdef VLA_TIMELINE
#define VLA_TL(tl, who, ev)                                                                          \
  do {                                                                                               \
    if ((tl) != nullptr && threadIdx.x == (who))                                                     \
      (tl)[((size_t)blockIdx.x + gridDim.x * (blockIdx.y + (size_t)gridDim.y * blockIdx.z)) * 16 + (ev)] = \
          VLA_TL_NOW();                                                                              \
  } while (0)
#else
#define VLA_TL(tl, who, ev) \
  do {                      \
  } while (0)
#endif

// ---------------------------------------------------------------------------
// Block reductions (blockDim.x a multiple of 32, <= 1024)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// `scratch` must hold 32 floats; all threads get the result.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[wid] = v;
  __syncthreads();
  float r = (lane < nw) ? scratch[lane] : 0.f;
  r = warp_sum(r);
  return r;
}
__device__ __forceinline__ float block_max(float v, float* scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) scratch[wid] = v;
  __syncthreads();
  float r = (lane < nw) ? scratch[lane] : 0.f;
  r = warp_max(r);
  return r;
}

// ---------------------------------------------------------------------------
// Eq. (4), first line, for one row held in shared memory by the whole block:
//   alpha = max(|x|_inf, 1e-5) / 127   (IEEE round-to-nearest division)
//   a_j   = clip(rint(x_j / alpha), -128, 127)   (rint: ties to even)
// Writes int8 codes (codes != nullptr) and/or the same integers as bf16
// carriers (carriers != nullptr; every |a| <= 128 is exact in bf16).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float quantize_row_block(const float* row, int K, int8_t* codes,
                                                    bf16* carriers, float* red_scratch) {
  float amax = 0.f;
  for (int i = threadIdx.x; i < K; i += blockDim.x) amax = fmaxf(amax, fabsf(row[i]));
  amax = block_max(amax, red_scratch);
  const float alpha = __fdiv_rn(fmaxf(amax, 1e-5f), 127.0f);
  for (int i = threadIdx.x; i < K; i += blockDim.x) {
    float r = rintf(__fdiv_rn(row[i], alpha));
    r = fminf(fmaxf(r, -128.f), 127.f);
    if (codes) codes[i] = (int8_t)(int)r;
    if (carriers) carriers[i] = __float2bfloat16_rn(r);
  }
  return alpha;
}

// Eq. (4), output line: bf16_rne((float(acc) * alpha) * beta), returned as fp32.
__device__ __forceinline__ float w2a8_scale(float acc, float alpha, float beta) {
  return __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(acc, alpha), beta)));
}

// Four ternary codes (one byte, code c_i = q_i + 1 in bits 2i..2i+1) as two
// bf16x2 words, element 0 in the low half of the first: a byte-permute table
// lookup.  Selector nibble i is c_i; the tables hold, for codes 0..3, the
// high bytes (BF 00 3F 00) and the low bytes (80 00 80 00) of -1, 0, +1, 0.
__device__ __forceinline__ uint2 ternary_quad_bf16(uint32_t byte) {
  const uint32_t sel = (byte & 0x3u) | ((byte & 0xCu) << 2) | ((byte & 0x30u) << 4) | ((byte & 0xC0u) << 6);
  uint32_t hi, lo, w0, w1;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(0x003F00BFu), "r"(0x00800080u), "r"(sel));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0x003F00BFu), "r"(0x00800080u), "r"(sel | 0x4444u));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(w0) : "r"(lo), "r"(hi), "r"(0x5140u));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(w1) : "r"(lo), "r"(hi), "r"(0x7362u));
  return make_uint2(w0, w1);
}

__device__ __forceinline__ float gelu_exact(float x) {
  return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
}

// Visibility bits of prefix keys [start, start + 32) of one observation from
// its mask row (nw words; bit p % 32 of word p / 32 set = key p visible, the
// additive mask M of Eq. (2) being 0 there and -inf elsewhere).  Keys past
// the row read as hidden; a null row is all visible.
__device__ __forceinline__ uint32_t prefix_mask_window(const uint32_t* row, int nw, int start) {
  if (!row) return 0xFFFFFFFFu;
  const int w = start >> 5, sh = start & 31;
  const uint32_t lo = (w >= 0 && w < nw) ? __ldg(row + w) : 0u;
  const uint32_t hi = (w + 1 >= 0 && w + 1 < nw) ? __ldg(row + w + 1) : 0u;
  return sh ? (lo >> sh) | (hi << (32 - sh)) : lo;
}

// ---------------------------------------------------------------------------
// PTX: shared-memory addresses, mbarriers, TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// shared to global memory, in the thread's bulk group.
__device__ __forceinline__ void bulk_store_s2g(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
// Commit the thread's bulk copies and wait until they have read their shared
// memory source (the writes to global memory complete with the grid).
__device__ __forceinline__ void bulk_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The status block a handle passes to its kernels: word 0 is the latched
// error, words 2-3 the bounded-wait limit in ns (0: the default limit; limits
// below 100 us act as 100 us).
__device__ __forceinline__ uint64_t wait_limit_ns(const int* status) {
  if (!status) return VLA_WAIT_LIMIT_NS;
  const uint64_t lim = *(const volatile unsigned long long*)(status + 2);
  return lim ? lim : VLA_WAIT_LIMIT_NS;
}
// Bounded wait for the phase with the given parity.  On timeout latches
// VLA_DEV_TIMEOUT and returns false; also gives up early once another thread
// has latched a timeout (the pipeline it belongs to is broken).  A latched
// abort does not end waits: every kernel of the launch runs to completion.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint64_t lim = 0;  // the handle's limit, read only once a wait has lasted 100 us
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    const uint64_t el = globaltimer_ns() - t0;
    if (el > 100000ull) {
      if (!lim) lim = wait_limit_ns(status);
      if (el > lim) {
        latch_error(status, VLA_DEV_TIMEOUT);
        return false;
      }
    }
    if (status && *(volatile int*)status == VLA_DEV_TIMEOUT) return false;
  }
}

// Bring the 128-byte line holding `p` into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}
// 2-D tiled TMA load into shared memory, completion via mbarrier tx bytes.
// x = innermost (contiguous) element coordinate, y = row.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const void* map, uint64_t* bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// PTX: thread-block clusters, distributed shared memory, programmatic
// dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA in the cluster; release/acquire orders the
// shared-memory writes before the barrier with the reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// Wait until the grids this one depends on (programmatic dependent launch)
// have completed and their memory is visible; a no-op without PDL.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the dependent grid start launching (its pre-wait prologue overlaps us).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Named barrier `id` (1..15) over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void st_shared_v4_u32(uint32_t saddr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// Two floats rounded to bf16 (nearest even) in one instruction; lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Byte offset of the 16-byte chunk `j` (0..7) of row `r` inside a K-major
// tile of 128-byte rows written with the 128-byte swizzle (the layout TMA
// produces with CU_TENSOR_MAP_SWIZZLE_128B and sdesc_k128 describes).
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t j) {
  return r * 128u + ((j ^ (r & 7u)) << 4);
}

// ---------------------------------------------------------------------------
// PTX: tcgen05 (5th-generation tensor cores, accumulators in TMEM)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, cta_group::1.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: the A operand read from tensor memory
// (row m in lane m, K along columns, two bf16 per 32-bit column, the lower K
// index in the low half), bf16 inputs, fp32 accumulate, cta_group::1.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 bit, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// tcgen05.ld of 16 columns without the wait: the raw registers must not be
// read until tmem_wait16() has run on them (that asm takes them as in/out
// operands, so the compiler cannot hoist a use above the wait).
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
// tcgen05.st of 16 columns (32 lanes x 32 bit); complete with tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Bounded wait that ignores the error latch: used only to let this CTA's own
// asynchronous copies or MMAs finish before it frees their destination.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > VLA_WAIT_LIMIT_NS) return;
}
// 2^x with the hardware approximation (relative error ~2^-22), for softmax.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory matrix descriptor (tcgen05 format) for a K-major operand tile
// whose rows are 128 bytes (64 bf16) with the 128-byte swizzle that TMA
// writes; 8-row core-matrix groups are 1024 bytes apart.  The tile base must
// be 1024-byte aligned; a K offset inside the row is added to the address.
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)0 << 16;                     // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                     // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}
// Instruction descriptor: kind::f16 with bf16 A/B, fp32 D, both K-major.
__host__ __device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// ---------------------------------------------------------------------------
// Host-side launch interfaces (implemented in the kernel translation units)
// ---------------------------------------------------------------------------
// K_C [L][B][n_kv][P][d_h]; V_C stored transposed [L][B][n_kv][d_h][P8].
struct KvScatter {
  void* kc;
  void* vc;
  int L, B, n_kv, P, d_h, P8;
};

struct DevCtl {
  int* status;               // latched device error word
  const volatile int* abort; // host-mapped abort flag (may be null)
};

// SIMT GEMM: out[z][t][n] = sum_{k in split z} X[t][k] W[n][k] (fp32 partials),
// or, when kv != nullptr, scatter D into K_C / V_C (1 split).
cudaError_t launch_gemm_simt(int x_bf16, const void* X, int ldx, int w_bf16, const void* W, int ldw, int T, int N,
                             int K, int splits, float* out, size_t split_stride, int ldo, const KvScatter* kv,
                             cudaStream_t st);

// tcgen05 GEMM with both operands K-major bf16 loaded by TMA:
// D[n][t] = sum_k W[a_row0 + n][k] * X[t][k]; A = weights (M = 128 rows per
// tile), B = tokens (BN rows per tile, 16 <= BN <= 256, BN % 16 == 0).
struct TcGemmArgs {
  int N;            // valid weight rows (output features)
  int T;            // valid token rows
  int a_row0;       // first weight row in the A tensor map (layer offset)
  int num_kb;       // K / 64
  int kb_per_split; // k-blocks per split (grid.z splits)
  int BN;           // token tile
  int stages;       // pipeline depth
  float* out;       // partial output [z][T][ldo] fp32 (kv == mode 0)
  size_t split_stride;
  int ldo;
  int mode;         // 0: fp32 partials; 1: K/V cache scatter (bf16)
  KvScatter kv;
  int* status;
};
int tc_encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows);
cudaError_t launch_gemm_tc(const CUtensorMap* tmA, const CUtensorMap* tmB, const TcGemmArgs& a, int tiles_n,
                           int tiles_t, int splits, cudaStream_t st);
size_t tc_smem_bytes(int BN, int stages);

// W2A8 SIMT ternary GEMM: out[z][t][n] = (float) sum_{k in split z} a[t][k] q[n][k]
// (exact integers), packed q [N][K/4].
cudaError_t launch_ternary_simt(const int8_t* a, int lda, const uint8_t* q, int T, int N, int K, int splits,
                                float* out, size_t split_stride, int ldo, cudaStream_t st);
cudaError_t launch_quantize_rows(const float* x, int M, int K, int8_t* a, float* alpha, cudaStream_t st);
cudaError_t launch_ternary_finish(const float* part, int M, int N, const float* alpha, float beta, uint16_t* y,
                                  int32_t* acc, cudaStream_t st);
cudaError_t launch_check_ternary_codes(const uint8_t* q, size_t nbytes, int* bad, cudaStream_t st);
// Split count that launch_gemm_simt / launch_ternary_simt actually use for a
// requested count (k range per split rounded up to `align`).
int simt_effective_splits(int K, int splits, int align);
// Raise a kernel's dynamic shared-memory limit to the device's opt-in
// maximum minus the kernel's static shared memory.
template <typename F>
inline cudaError_t set_max_dyn_smem(F* func) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, (const void*)func);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void*)func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes);
  return e;
}
// Records the failing CUDA call for vla_last_error().
void vla_set_last_error(const char* where, cudaError_t e);

// One-time kernel attribute set-up (dynamic shared memory limits); call
// before any stream capture.
cudaError_t simt_kernels_init();
cudaError_t tc_kernels_init();
cudaError_t expert_kernels_init();
cudaError_t launch_to_f32(const void* src, int src_bf16, float* dst, size_t n, cudaStream_t st);

// Fused cluster split-K linear layer (k_linear_tc.cu).
enum { EPI_QKV = 0, EPI_RESID = 1, EPI_GELU = 2, EPI_W2A8_OUT = 3, EPI_KV = 4 };
struct LinArgs {
  int N;        // output features (weight rows), multiple of 4
  int T;        // tokens
  int a_row0;   // first weight row in the A tensor map (layer offset)
  int KS;       // K range per cluster rank (multiple of 64); K = C * KS
  int BN;       // token tile, 16..256, multiple of 16
  int stages;   // weight ring depth
  int bmode;    // 0: B tiles by TMA (tmB over [T][K] bf16); 1: B = modulated RMSNorm of h
  int amode;    // 0: A (weights) bf16 by TMA; 1: packed 2-bit ternary codes by TMA, decoded to bf16 in smem
                // (a ring of `stages` code stages); 2: the same with every k-block's codes loaded at once
                // (KS / 64 <= 16)
  int epi;      // EPI_*
  // W2A8 (Eq. 4): the accumulators are exact integers; y = bf16((acc * alpha_t) * beta)
  int w2a8;
  const float* alpha;  // [T] per-token activation scales
  const float* wbeta;  // per-output-row weight scales beta_{g(n)}: row n of this map at
                       // wbeta[layer * beta_stride + beta_off + n]; null: beta_val for every row
  float beta_val;
  int layer;
  int beta_stride, beta_off;
  float* g32;          // EPI_GELU with W2A8: fp32 GeLU output [T][ldg] (quantised next)
  uint16_t* yout;      // EPI_W2A8_OUT: bf16 bits [T][N]
  int32_t* accout;     // EPI_W2A8_OUT: int32 accumulators [T][N] (nullable)
  // bmode 1 inputs
  const float* h_in;   // [T][D] residual stream
  const float* ss_in;  // [n_ss_in][T] partial sums of squares of h rows
  int n_ss_in;
  const float* gamma;  // [D]
  const float* beta;   // [D]
  float eps;
  int D;               // width of h (row pitch of h / h_in)
  // EPI_RESID
  float* h;            // [T][D]
  float* ss_out;       // [tiles_n][T]: sums of squares of each 128-row block (nullptr: not needed)
  // EPI_GELU
  bf16* g;
  int ldg;
  // EPI_QKV
  bf16* q;             // [B][n_q][H][d_h]
  bf16* ks;            // [B][n_kv][H][d_h]
  bf16* vst;           // [B][n_kv][d_h][Hp]
  int H, n_q, n_kv, d_h, qdim, kvdim, Hp;
  // EPI_KV (prefix K/V cache build, Eq. 2): rows [L][K|V][n_kv][d_h], tokens [B][P]
  bf16* kc_out;  // K_C [L][B][n_kv][P][d_h]
  bf16* vc_out;  // V_C^T [L][B][n_kv][d_h][P8]
  int kv_B, kv_P, kv_P8;
  // split-K exchange through L2: [tile][rank][BN][128] fp32 partials and
  // [tile][rank][BN] per-token sums of squares (tile = tile_t * tiles_n + tile_n)
  float* xpart;
  float* xss;
  int* status;
  unsigned long long* tl;  // event trace (VLA_TIMELINE builds), else unused
  // Factored modulated RMSNorm (many-token kernel only).  With
  // u = h r (1 + gamma) + beta and r = 1 / rms(h):  W u = r W ((1 + gamma) h) + W beta.
  // EPI_RESID: xt_out (nullable) [T][D] bf16 receives (1 + xt_gamma[n]) h_new,
  // the operand of the next normed map.  EPI_QKV / EPI_GELU: if fn_c is set,
  // the B operand is that scaled h, and y = r_t acc + fn_c[n], with r_t from the
  // fn_nss per-block sums of squares fn_ss [fn_nss][T].
  bf16* xt_out;
  const float* xt_gamma;  // [D]
  // EPI_RESID, cluster split: each rank writes its own rows' per-token sums of
  // squares to slot (tile_n * C + rank) of ss_out instead of combining the
  // ranks' sums behind a second cluster barrier (the consumer sums the
  // slots, in fixed order)
  int ss_per_rank;
  const float* fn_c;      // [N]  W beta of this (step, layer)
  const float* fn_ss;
  int fn_nss;
};
size_t linear_smem_bytes(const LinArgs& g);
cudaError_t linear_kernels_init();
// tmH: fp32 map over h [T][D] with box 64 x BN (no swizzle), used by bmode 1.
cudaError_t launch_linear(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmH, const LinArgs& g,
                          int tiles_n, int tiles_t, int C, cudaStream_t st);

// cudaError_t launch_linear also takes EPI_KV with packed ternary weights
// (AMODE 1, no split): the W2A8 prefix cache build.

// Persistent many-token linear kernel (k_linear_wide.cu): same LinArgs and
// epilogues (EPI_QKV, EPI_RESID, EPI_GELU, and EPI_KV for the prefix K/V
// build; bf16 weights, TMA'd tokens with a 64 x BN box, KS = K), BN a
// multiple of 16 in [64, 256], N a multiple of 128.
size_t linear_wide_smem_bytes(int BN);
// GeLU by erff and by the many-token epilogue's approximation, elementwise.
cudaError_t launch_gelu_forms(const float* x, int n, float* exact, float* fast, cudaStream_t st);
cudaError_t linear_wide_init();
cudaError_t launch_linear_wide(const CUtensorMap* tmA, const CUtensorMap* tmB, const LinArgs& g, int grid,
                               cudaStream_t st);

// tcgen05 joint attention (k_attn_tc.cu): a cluster of `cs` CTAs per
// 128-row query tile of one (observation, K/V head); ranks 0..cs-2 take kc
// prefix keys each, rank cs-1 the action keys; merged on chip into o.
struct AttnArgs {
  int B, P, H, n_q, n_kv, d_h, group;  // group = n_q / n_kv
  int layer;
  int n_qt;          // query tiles per (observation, K/V head)
  int cs;            // cluster size (power of two, 2..16)
  int kc;            // prefix keys per rank (multiple of 16, <= 128)
  int kc_s;          // action-key tile (H rounded up to 16, <= 128)
  float scale_log2;  // log2(e) / sqrt(d_h)
  bf16* o;           // [B*H][n_q*d_h] output
  const uint32_t* pmask;  // prefix visibility bits [B][pmw] (null: every prefix key visible)
  int pmw;                // mask words per observation, (P + 31) / 32
  int no_suffix;          // a cross-attention layer: the cached keys only, no action keys
  bf16* xo;          // L2 exchange of unnormalised partial O: [tile][rank][d_h/8][128][8] bf16
  float2* xml;       // and of each partial's row maximum and sum (m, l): [tile][rank][128]
  float* o32;        // when set, o is written in fp32 here instead of bf16 (W2A8 quantises it next)
  int* status;
  unsigned long long* tl;  // event trace (VLA_TIMELINE builds), else unused
};
size_t attn_tc_smem_bytes(int d_h, int kc);
cudaError_t attn_kernels_init();
// tmQ over q [B*n_q*H][d_h] (box 64 x 128); tmK over K_C {d_h, P, L*B*n_kv}
// (box 64 x kc); tmVt over V_C^T {P, d_h, L*B*n_kv} (box 64 x d_h); tmKs over
// k_s {d_h, H, B*n_kv} (box 64 x kc_s); tmVs over v_s^T {H, d_h, B*n_kv}
// (box 64 x d_h); all bf16 with the 128-byte swizzle.
cudaError_t launch_attn_tc(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmVt,
                           const CUtensorMap* tmKs, const CUtensorMap* tmVs, const AttnArgs& a, cudaStream_t st);
// Streaming joint attention (k_attn_stream.cu): one CTA per 128-row query
// tile streams every key in 128-key chunks (no cross-CTA merge).  Uses the
// AttnArgs fields B, P, H, n_q, n_kv, d_h, group, layer, n_qt, scale_log2, o,
// o32, status.  tmK and tmKs have 128-row boxes; tmQ, tmVt, tmVs as above.
size_t attn_stream_smem_bytes(int d_h);
cudaError_t attn_stream_init();
cudaError_t launch_attn_stream(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmVt,
                               const CUtensorMap* tmKs, const CUtensorMap* tmVs, const AttnArgs& a, cudaStream_t st);
int tc_encode_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                     uint32_t box_rows);
// uint8 map (no swizzle) over packed ternary codes [rows][inner bytes].
int tc_encode_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows);
int tc_encode_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                      uint64_t stride2_bytes, uint32_t box0, uint32_t box1);

// Persistent whole-solve kernel for few tokens (k_solver_persist.cu).
struct PersistArgs {
  int L, D, F, S, T, BN, B, H, Hp, P, d_a, d_h, n_q, n_kv, group, qdim, kvdim, qkvdim;
  int n_att;                      // attention CTAs (the last n_att of the grid)
  int nqt, npch, nch, att_units;  // query tiles per (b, g), cached-key chunks, all chunks, units
  int U[4], nkb[4], N[4];         // linear phases (qkv, o, up, down): units, K blocks, rows
  int work_bytes;                 // linear CTAs' operand + staging region
  float eps, scale_log2, dt_sign;
  const float* win;     // [D][d_a]
  const float* wout;    // [d_a][D]
  const float* modtab;  // [S][L][4][D]
  const float* modf;    // [S][2][D]
  const float* cqkv;    // [S][L][qkvdim]  W_qkv beta_a
  const float* cup;     // [S][L][F]       W_up beta_m
  const float* noise;   // [T][d_a]
  float* actions;       // [T][d_a]
  float* vtap;          // [S][T][d_a] or null
  float* h;             // [T][D]
  float* accq;          // [T][qkvdim]
  float* accu;          // [T][F]
  float* rms;           // [2][T]
  bf16* q;              // [B][n_q][H][d_h]
  bf16* ks;             // [B][n_kv][H][d_h]
  bf16* vs;             // [B][n_kv][d_h][Hp]
  bf16* o;              // [T][qdim]
  float* opart;         // [B*n_kv*nch][group*H][d_h] unnormalised chunk outputs
  float2* oml;          // [B*n_kv*nch][group*H]
  unsigned* bar;        // grid barrier counter; bar[1] is the stop word
  int* stop;
  int* status;
  const volatile int* abort;
  const uint32_t* pmask;      // prefix visibility bits [B][pmw] (null: all visible)
  int pmw;
  unsigned long long* trace;  // phase trace (-DVLA_PERSIST_TRACE builds), else unused
};
size_t persist_smem_bytes(int D);
int persist_ring_stages(int D, int work_bytes);
bool persist_att_fits(int dh);
cudaError_t persist_init();
cudaError_t persist_blocks_per_sm(int D, int* n);
// maps[15]: bf16 weights [W_q;W_k;W_v], W_o, W_up, W_down (box 64 x 128);
// K_C {d_h, P, L*B*n_kv} (box 64 x 128); V_C^T {P, d_h, L*B*n_kv} (box 64 x
// d_h); k_s {d_h, H, B*n_kv} (box 64 x 128); v_s^T {H, d_h, B*n_kv} (box 64 x
// d_h); q [B*n_q*H][d_h] (box 64 x 128); h and acc_up fp32 (box 64 x BN, no
// swizzle); o bf16 (box 64 x BN); acc_qkv, h, acc_up fp32 (box 128 x BN, no
// swizzle) for the reductions.  Clears the barrier words, then one
// cooperative launch of `grid` CTAs.
cudaError_t launch_persist(const CUtensorMap* maps, const PersistArgs& a, int grid, cudaStream_t st);

// Expert kernels (k_expert.cu).
struct ExpertDims {
  int L, D, F, n_q, n_kv, d_h, d_a, H, B, P, S, d_t;
  int P8;  // P rounded up to a multiple of 8: row pitch of V_C^T
  int Hp;  // H rounded up to a multiple of 8: row pitch of v_s^T
  float eps;
  int qdim, kvdim, qkvdim;
  int f32;   // 1 when the config dtype is fp32
  int w2a8;  // 1 for the ternary / int8 variant
};

struct StepBufs {
  // weights
  const float* win;     // [D][d_a]
  const float* wout;    // [d_a][D]
  const float* modtab;  // [S][L][4][D]
  const float* modf;    // [S][2][D]
  const float* beta;    // [L][6] (W2A8)
  // workspace
  float* h;             // [T][D]
  void* act;            // [T][Kmax] GEMM input (bf16 / fp32 / bf16 carriers)
  int8_t* codes;        // [T][Kmax] W2A8 int8 codes (SIMT ternary path)
  float* alpha;         // [T] W2A8 row scales
  float* part;          // [splits][T][N] GEMM partials
  void* q;              // [B][n_q][H][d_h]
  void* ks;             // [B][n_kv][H][d_h]
  void* vs;             // [B][n_kv][d_h][Hp] (transposed)
  float* opart;         // attention partial outputs
  float* ml;            // attention partial (max, sum)
  int attn_chunk, n_chunks;
  const uint32_t* pmask;  // prefix visibility bits [B][pmw] (null: all visible)
  int pmw;
  int no_suffix;          // attention of a cross-attention layer: cached keys only
};

// tau_k = k / S, or 1 - k / S when reverse.
cudaError_t launch_time_embed(float* e, int S, int d_t, int reverse, cudaStream_t st);
// n normals of the seeded Philox4x64-10 / Box-Muller stream (X^0).
cudaError_t launch_noise(unsigned long long seed, size_t n, float* out, cudaStream_t st);
cudaError_t launch_silu(float* x, size_t n, cudaStream_t st);
cudaError_t launch_embed_norm(const ExpertDims& d, const StepBufs& b, int step, const float* x_in, DevCtl ctl,
                              cudaStream_t st);
cudaError_t launch_reduce_qkv(const ExpertDims& d, const StepBufs& b, int layer, int splits, cudaStream_t st);
cudaError_t launch_attention(const ExpertDims& d, const StepBufs& b, int layer, const void* kc, const void* vc,
                             cudaStream_t st);
size_t attention_smem_bytes(const ExpertDims& d, int chunk);
cudaError_t launch_reduce_norm(const ExpertDims& d, const StepBufs& b, int step, int layer_for_beta,
                               int beta_slot, int mod_layer, int mod_half, int splits, cudaStream_t st);
cudaError_t launch_reduce_gelu(const ExpertDims& d, const StepBufs& b, int layer, int splits, cudaStream_t st);
cudaError_t launch_head(const ExpertDims& d, const StepBufs& b, int step, int splits, float dt, const float* x_in,
                        float* x_out, float* tap, cudaStream_t st);
// Fused-path helpers: h = x W_in^T with its row sums of squares (1 slot);
// u = modulated RMSNorm of h as bf16 [T][D] (for token tiles too large for
// the in-GEMM prologue); the velocity head reading h directly.
// xt (nullable) also receives bf16((1 + xgam) h) (factored modulated norm).
cudaError_t launch_embed_ss(const ExpertDims& d, const StepBufs& b, const float* x_in, float* ss_out, DevCtl ctl,
                            cudaStream_t st, bf16* xt = nullptr, const float* xgam = nullptr);
// Sum-of-squares slots k_embed_ss / k_embed_ss_multi write for this shape.
int embed_ss_slots(const ExpertDims& d);
cudaError_t launch_modnorm(const ExpertDims& d, const float* h, const float* ss, int n_ss, const float* gamma,
                           const float* beta, bf16* u, cudaStream_t st);
cudaError_t launch_head_fused(const ExpertDims& d, const StepBufs& b, int step, float dt, const float* x_in,
                              float* x_out, float* tap, cudaStream_t st);
// W2A8 row quantisers (Eq. 4): bf16 carriers of the int8 codes [T][K] and
// alpha [T].  quant_norm quantises the modulated RMSNorm of h (computing the
// row's rms itself); quant_rows quantises fp32 rows x [T][K].
// u_out (nullable): the fp32 modulated rows that were quantised [T][D].
cudaError_t launch_quant_norm(const ExpertDims& d, const float* h, const float* gamma, const float* beta, bf16* codes,
                              float* alpha, float* u_out, cudaStream_t st);
cudaError_t launch_quant_rows(int T, int K, const float* x, bf16* codes, float* alpha, cudaStream_t st);
// The same quantiser writing int8 codes (the standalone Eq. (4) entry point).
cudaError_t launch_quant_rows_i8(int T, int K, const float* x, int8_t* codes, float* alpha, cudaStream_t st);
// Eq. (4) on bf16 rows (W2A8 prefix build): bf16 carriers of the codes and alpha.
cudaError_t launch_quant_rows_bf16(int T, int K, const bf16* x, bf16* codes, float* alpha, cudaStream_t st);
// dst[l * stride + off + n] = src[l * (N / G) + n / G] for n < N, l < L.
cudaError_t launch_expand_scales(float* dst, const float* src, int L, int N, int G, int stride, int off,
                                 cudaStream_t st);
// Sets *bad unless every row of idx [L][Fs] is strictly increasing in [0, F).
cudaError_t launch_check_ffn_idx(const int32_t* idx, int L, int F, int Fs, int* bad, cudaStream_t st);
// Compact W_up rows / W_down columns of the selected FFN neurons idx [L][Fs].
cudaError_t launch_gather_ffn(const bf16* wup, const bf16* wdown, bf16* up_sel, bf16* down_sel, const int32_t* idx,
                              int L, int F, int D, int Fs, cudaStream_t st);
// One kernel whose bounded wait cannot be satisfied (exercises the timeout latch).
cudaError_t launch_expire_wait(int* status, cudaStream_t st);
cudaError_t launch_i8_to_bf16(const int8_t* a, bf16* out, size_t n, cudaStream_t st);

