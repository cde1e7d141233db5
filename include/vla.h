/*
 * vla.h - C ABI of libvla, the GB300 (sm_103a) library for the hot path of
 * flow-matching vision-language-action inference with a prefix K/V cache.
 *
 * Source of the operations: "vla.cpp: A Unified Inference Runtime for
 * Vision-Language-Action Models":
 *   - §III-A, Eq. (1): Euler integration of an action chunk
 *       X^{k+1} = X^k + (tau_{k+1} - tau_k) v(X^k, tau_k, C)
 *     from noise X^0 in R^{H x d_a} over T solver steps (here n_steps = S).
 *   - §III-B, Eq. (2): the observation prefix Z is projected once per
 *     observation into per-layer keys/values K_C = Z W_K, V_C = Z W_V, reused
 *     by every solver step (cache lifecycle: refreshed per observation, reused
 *     within a request); the action tokens attend to [K_C ; own keys] with
 *     softmax(Q K^T / sqrt(d_k) + M) V (joint attention; M = 0 unless a
 *     request hides prefix keys, see vla_request).
 *   - §III-D, Eq. (4): ternary weights (four 2-bit codes per byte, fp32
 *     scales beta_{g(n)} per tensor or per group of output rows) with per-row
 *     int8 activations, 32-bit integer accumulation and bf16 output.
 *   - §III-C: requests carry inputs and optional noise and masks; responses
 *     carry the action chunk and its dimensions, or an error.
 *
 * Conventions for every call:
 *   - Pointers named *_dev are DEVICE pointers owned by the caller; the
 *     library never frees them.  Pointers named *_host are host pointers.
 *     Every tensor pointer must be 16-byte aligned.
 *   - Weights are stored out-major: a map R^in -> R^out is [out][in] with
 *     `in` contiguous (y = x W^T).  Stacked per-layer weights are [L][out][in].
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work on it and return without synchronising
 *     unless stated otherwise.
 *   - Argument and shape errors are returned synchronously before anything is
 *     enqueued.  Errors raised on the device (a bounded wait that timed out)
 *     are latched in the handle and returned by vla_expert_poll_status().
 *   - A handle is not re-entrant: one call in flight per handle.
 */
#ifndef VLA_H_
#define VLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VLA_OK = 0,
  VLA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad enum, B or P out of range */
  VLA_ERR_SHAPE = 2,        /* inconsistent dimensions */
  VLA_ERR_UNSUPPORTED = 3,  /* valid but not implemented (e.g. K not a multiple of 64 for bf16) */
  VLA_ERR_OOM = 4,          /* device allocation failed */
  VLA_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  VLA_ERR_TIMEOUT = 6,      /* a device-side bounded wait gave up (latched) */
  VLA_ERR_ABORTED = 7,      /* a kernel saw the handle's abort flag (latched) */
  VLA_ERR_NO_DEVICE = 8     /* no usable sm_103 device */
} vla_status;

typedef enum { VLA_DTYPE_F32 = 0, VLA_DTYPE_BF16 = 1 } vla_dtype;

/* Time convention of the solver schedule (§III-A): FORWARD integrates
 * tau_k = k / S from 0 to 1 (GR00T); REVERSE integrates tau_k = 1 - k / S from
 * 1 to 0 (SmolVLA, pi0): the network is evaluated at the reversed time and the
 * velocity sign change enters Eq. (1) through tau_{k+1} - tau_k = -1/S. */
typedef enum { VLA_SCHEDULE_FORWARD = 0, VLA_SCHEDULE_REVERSE = 1 } vla_schedule;

/* Diagnostic flags for vla_expert_config.flags. */
#define VLA_FLAG_SIMT_GEMM 1u  /* run bf16 GEMMs on the CUDA-core kernel instead of tcgen05 */
#define VLA_FLAG_NO_GRAPH 2u   /* enqueue the solver kernels directly instead of one graph launch */
#define VLA_FLAG_ATTN_SPLIT 4u  /* attention: always the clustered form (a query tile's keys split over SMs;
                                   it holds at most 1920 prefix keys, and at most 896 when d_h is 64 or 192: beyond
                                   that the call fails, while without this flag such prefixes take the
                                   streaming form where d_h is 64, 128 or 256) */
#define VLA_FLAG_ATTN_STREAM 8u /* attention: the streaming form (one CTA per query tile, all keys) where d_h is 64, 128 or 256 */
#define VLA_FLAG_LINEAR_SPLIT 16u /* bf16 linear layers: always the cluster split-K kernel */
#define VLA_FLAG_LINEAR_WIDE 32u  /* bf16 linear layers: the persistent many-token kernel wherever N % 128 == 0 */
#define VLA_FLAG_PERSIST 64u      /* few tokens (bf16, B*H <= 64): the whole solve as one persistent cooperative kernel */

typedef struct {
  int n_layers;    /* L */
  int width;       /* D, expert hidden width */
  int mlp_width;   /* F */
  int n_q_heads;   /* n_q */
  int n_kv_heads;  /* n_kv; n_q % n_kv == 0, query head j reads K/V head j / (n_q / n_kv) */
  int head_dim;    /* d_h (= d_k of Eq. 2) */
  int vlm_hidden;  /* d_vlm, width of the prefix hidden states Z */
  int action_dim;  /* d_a */
  int horizon;     /* H, actions per chunk */
  int time_dim;    /* d_t, sinusoidal time embedding width (even) */
  int max_batch;   /* largest B any call will use; sizes the workspace */
  int max_prefix;  /* largest P any call will use */
  int dtype;       /* vla_dtype of weights, Z and the K/V cache (W2A8: BF16) */
  float rms_eps;   /* RMSNorm epsilon (1e-6) */
  unsigned flags;  /* VLA_FLAG_* (0 for normal use) */
  int schedule;    /* vla_schedule */
  int cross_every; /* 0: every layer is joint attention over [K_C ; action keys]; k > 0: layers l with
                      l mod k == k - 1 are cross-attention layers whose queries see the cached prefix
                      keys only (the alternating joint / cross design, §III-B); their W_k, W_v rows
                      are unused.  A prefix mask must then leave each observation a visible key. */
} vla_expert_config;

/* Dense weights, device pointers of the config dtype, shapes [..][out][in]. */
typedef struct {
  const void* wk_pre;  /* [L][n_kv*d_h][d_vlm]  W_K of Eq. 2, per layer */
  const void* wv_pre;  /* [L][n_kv*d_h][d_vlm]  W_V of Eq. 2, per layer */
  const void* wq;      /* [L][n_q*d_h][D] */
  const void* wk;      /* [L][n_kv*d_h][D]   action-token keys */
  const void* wv;      /* [L][n_kv*d_h][D]   action-token values */
  const void* wo;      /* [L][D][n_q*d_h] */
  const void* wup;     /* [L][F][D] */
  const void* wdown;   /* [L][D][F] */
  const void* wmod;    /* [L][4D][D]  -> (gamma_a, beta_a, gamma_m, beta_m) */
  const void* win;     /* [D][d_a]    action in-projection */
  const void* wout;    /* [d_a][D]    velocity projection */
  const void* wt1;     /* [D][d_t]    time MLP, first map */
  const void* wt2;     /* [D][D]      time MLP, second map */
  const void* wmod_f;  /* [2D][D]     -> (gamma_f, beta_f) of the final norm */
} vla_expert_weights;

/* W2A8 weights: the six per-layer maps W_q, W_k, W_v, W_o, W_up, W_down are
 * ternary, packed uint8 [L][out][in/4] (code q+1 of input index j at bits
 * 2*(j mod 4) of byte j/4; code 3 is invalid), each with fp32 scales
 * beta_{g(n)} of Eq. (4): with beta_group == 0 one scale per tensor and layer
 * ([L] floats), else one per group of beta_group consecutive output rows
 * ([L][out / beta_group] floats; beta_group must divide every map's rows, a
 * multiple of 4).  The prefix maps are bf16 (wk_pre, wv_pre) unless
 * wk_pre_t / wv_pre_t are given: then they are ternary too ([L][n_kv*d_h]
 * [d_vlm/4], scales beta_wk_pre / beta_wv_pre grouped like the others, wk_pre
 * and wv_pre ignored) and vla_prefix_kv_build quantises each prefix row of Z
 * per Eq. (4) before the ternary product.  Everything else is bf16. */
typedef struct {
  const void* wk_pre;
  const void* wv_pre;
  const uint8_t* wq;
  const uint8_t* wk;
  const uint8_t* wv;
  const uint8_t* wo;
  const uint8_t* wup;
  const uint8_t* wdown;
  const float* beta_wq;
  const float* beta_wk;
  const float* beta_wv;
  const float* beta_wo;
  const float* beta_wup;
  const float* beta_wdown;
  const void* wmod;
  const void* win;
  const void* wout;
  const void* wt1;
  const void* wt2;
  const void* wmod_f;
  int beta_group;          /* 0: per-tensor scales; else output rows per scale group */
  const uint8_t* wk_pre_t; /* NULL, or ternary prefix W_K [L][n_kv*d_h][d_vlm/4] */
  const uint8_t* wv_pre_t; /* NULL, or ternary prefix W_V (both or neither) */
  const float* beta_wk_pre;
  const float* beta_wv_pre;
} vla_expert_weights_w2a8;

typedef struct vla_expert vla_expert;

/* Create an expert handle for a fixed solver length n_steps = S with the
 * uniform schedule of cfg->schedule (tau_k = k / S, dt = 1/S; or reverse).
 * Copies and repacks the weights into handle-owned device memory (the caller
 * may free its copies once the call returns), precomputes the time
 * conditioning table for every tau_k, and allocates the workspace for
 * max_batch x horizon action tokens, so that no later call allocates (except
 * the first vla_policy_step_host, see there).  Synchronises `stream`.
 * Returns VLA_ERR_INVALID_ARG / VLA_ERR_SHAPE / VLA_ERR_UNSUPPORTED for bad
 * configs, VLA_ERR_OOM, VLA_ERR_CUDA, VLA_ERR_NO_DEVICE. */
vla_status vla_expert_create(const vla_expert_config* cfg, const vla_expert_weights* w,
                             int n_steps, void* stream, vla_expert** out);

/* Same for the W2A8 variant (cfg->dtype must be VLA_DTYPE_BF16).  A packed
 * byte holding code 3 is rejected with VLA_ERR_INVALID_ARG. */
vla_status vla_expert_create_w2a8(const vla_expert_config* cfg, const vla_expert_weights_w2a8* w,
                                  int n_steps, void* stream, vla_expert** out);

/* Synchronises the device and frees everything the handle owns.  NULL is a no-op. */
void vla_expert_destroy(vla_expert* h);

/* Bytes to allocate for EACH of the two cache tensors for (B, P):
 * L * B * n_kv * P8 * d_h * sizeof(dtype), P8 = P rounded up to a multiple
 * of 8 (K_C needs only L * B * n_kv * P * d_h of it). */
vla_status vla_prefix_cache_bytes(const vla_expert* h, int B, int P, size_t* bytes_per_tensor);

/* Eq. 2, once per observation: K_C^l = Z W_K^l, V_C^l = Z W_V^l for every layer.
 *   Z_dev   [B][P][d_vlm]            config dtype, read only
 *   Kc_dev  [L][B][n_kv][P][d_h]     config dtype, written
 *   Vc_dev  [L][B][n_kv][d_h][P8]    config dtype, written: V_C stored
 *           transposed, P8 = P rounded up to a multiple of 8 (each row of
 *           V_C^T starts 16-byte aligned; entries p >= P are not written)
 * 1 <= B <= max_batch, 1 <= P <= max_prefix.  No mask and no positions enter
 * the projection.  Enqueues one kernel. */
vla_status vla_prefix_kv_build(vla_expert* h, const void* Z_dev, int B, int P,
                               void* Kc_dev, void* Vc_dev, void* stream);

/* Eq. 1 over S solver steps, reusing the cache of vla_prefix_kv_build.
 *   Kc_dev, Vc_dev   the cache for the same (B, P), read only
 *   noise_dev        [B][H][d_a] fp32, X^0 (required; NULL -> VLA_ERR_INVALID_ARG)
 *   actions_dev      [B][H][d_a] fp32, receives X^S (may alias noise_dev)
 *   vel_tap_dev      NULL or [S][B][H][d_a] fp32, receives every v_k
 * Every step evaluates the velocity network (time-modulated RMSNorm, joint
 * GQA attention over [K_C ; action keys], GeLU MLP, velocity projection) and
 * applies x <- x + dt v.  The S-step loop is one CUDA-graph launch (built on
 * the first call for a given (B, P, pointers) and reused afterwards). */
vla_status vla_action_denoise(vla_expert* h, const void* Kc_dev, const void* Vc_dev, int B, int P,
                              const float* noise_dev, float* actions_dev, float* vel_tap_dev,
                              void* stream);

/* The same solver with the W2A8 maps (handle from vla_expert_create_w2a8);
 * every ternary map quantises its input rows per Eq. 4 first. */
vla_status vla_action_denoise_w2a8(vla_expert* h, const void* Kc_dev, const void* Vc_dev, int B,
                                   int P, const float* noise_dev, float* actions_dev,
                                   float* vel_tap_dev, void* stream);

/* Per-request options (§III-C: requests carry inputs plus optional noise and
 * masks):
 *   prefix_mask_dev  NULL (every cached key visible) or uint32 [B][(P+31)/32]
 *                    device bits: bit p % 32 of word p / 32 of observation b
 *                    set = prefix key p visible (M = 0 in Eq. 2), clear =
 *                    hidden (M = -inf).  The action tokens' own keys are always
 *                    visible, so every query row keeps at least one key.  4-byte
 *                    aligned.  A per-observation prefix length P_b is the mask
 *                    with bits [0, P_b) set.
 *   noise_dev        X^0 [B][H][d_a] fp32, or NULL: the library draws X^0 ~ N(0, I)
 *                    from `seed` (vla_noise_fill's stream) into a handle-owned
 *                    buffer (allocated by the first such call)
 *   seed             the Philox key when noise_dev is NULL
 *   noise_out_dev    NULL, or [B][H][d_a] fp32 receiving the drawn X^0 */
typedef struct {
  const uint32_t* prefix_mask_dev;
  const float* noise_dev;
  unsigned long long seed;
  float* noise_out_dev;
} vla_request;

/* Eq. 1 with the per-request options above; dense or W2A8 by the handle.
 * Otherwise as vla_action_denoise (one graph launch per (B, P, pointers,
 * mask)). */
vla_status vla_action_denoise_ex(vla_expert* h, const void* Kc_dev, const void* Vc_dev, int B, int P,
                                 const vla_request* req, float* actions_dev, float* vel_tap_dev, void* stream);

/* n standard normals into out_dev (fp32): element e is normal (e mod 4) of
 * Philox4x64-10 block e / 4 (Salmon et al., SC 2011) under key (seed, 0) and
 * counter (e / 4, 0, 0, 0); words (x0, x1) and (x2, x3) of a block each give
 * two normals by the Box-Muller transform in fp64:
 * sqrt(-2 ln u1) (cos 2 pi u2, sin 2 pi u2), u1 = ((x0 >> 11) + 1) 2^-53,
 * u2 = (x1 >> 11) 2^-53.  The noise the solver draws for a request is this
 * stream over [B][H][d_a]. */
vla_status vla_noise_fill(unsigned long long seed, size_t n, float* out_dev, void* stream);

/* One whole request from host memory: copies Z and the noise to the device,
 * builds the prefix cache, runs the solver and copies X^S back, then
 * synchronises `stream`.  Z_host [B][P][d_vlm] (config dtype), noise_host and
 * actions_host [B][H][d_a] fp32; pinned host memory gives asynchronous
 * copies.  The first call allocates handle-owned device buffers for
 * max_batch x max_prefix (kept until destroy); later calls allocate nothing. */
vla_status vla_policy_step_host(vla_expert* h, const void* Z_host, int B, int P,
                                const float* noise_host, float* actions_host, void* stream);

/* Synchronises `stream` and returns the first error latched on the device
 * since the last poll (VLA_ERR_TIMEOUT, VLA_ERR_ABORTED) or VLA_OK; clears it. */
vla_status vla_expert_poll_status(vla_expert* h, void* stream);

/* Sets (1) or clears (0) the handle's abort flag (host-mapped memory, no
 * device call).  The first kernel of every solver step reads it; if it is
 * set, VLA_ERR_ABORTED is latched and vla_expert_poll_status() reports it.
 * The launch in flight runs to completion (bounded; no kernel is cut off with
 * work outstanding), and the action chunk of an aborted call is unspecified.
 * Clear the flag and poll the status before the next request. */
vla_status vla_expert_set_abort(vla_expert* h, int abort);

/* Limit, in ns, of every bounded device-side wait of this handle's kernels
 * (a wait that runs out latches VLA_ERR_TIMEOUT, frees what its CTA holds and
 * returns).  0 restores the default of 2 s.  Synchronous (a small host to
 * device copy); applies to kernels enqueued after the call. */
vla_status vla_expert_set_wait_limit(vla_expert* h, unsigned long long limit_ns);

/* Failure-path check: enqueues one single-thread kernel whose bounded wait can
 * never be satisfied (an mbarrier expecting two arrivals gets one).  The wait
 * runs out after the handle's wait limit, latches VLA_ERR_TIMEOUT and the
 * kernel returns with nothing left in flight; vla_expert_poll_status() then
 * returns VLA_ERR_TIMEOUT (and clears it) and the handle stays usable. */
vla_status vla_expert_check_wait_timeout(vla_expert* h, void* stream);

/* Diagnostic tap of the W2A8 solver (§III-E of the paper: intermediate
 * tensors localize discrepancies).  While a tap is set, W2A8 denoise calls on
 * this handle run without the CUDA graph and record, for solver step `step`,
 * every layer's intermediate tensors into tap_dev; NULL clears the tap.
 * tap_dev needs vla_expert_w2a8_tap_bytes(h, max_batch) bytes.  For batch B
 * (T = B*H tokens, Q = n_q*d_h, QKV = Q + 2*n_kv*d_h, Hp = H rounded up to a
 * multiple of 8), layer l's record starts at l * (bytes / L) and holds, in
 * this order, each tensor starting on a 256-byte boundary:
 *    0 h_in   f32  [T][D]    residual stream entering the layer
 *    1 u_a    f32  [T][D]    modulated RMSNorm (attention), the quantiser input
 *    2 c_a    bf16 [T][D]    its Eq. 4 codes (integers carried in bf16)
 *    3 al_a   f32  [T]       their row scales alpha
 *    4 acc_qkv i32 [T][QKV]  exact accumulators of [W_q;W_k;W_v]
 *    5 q      bf16 [B][n_q][H][d_h]
 *    6 k_s    bf16 [B][n_kv][H][d_h]
 *    7 v_s^T  bf16 [B][n_kv][d_h][Hp]
 *    8 o      f32  [T][Q]    attention output (quantiser input)
 *    9 c_o    bf16 [T][Q]   10 al_o f32 [T]   11 acc_o i32 [T][D]
 *   12 h_mid  f32  [T][D]    after the O-projection residual
 *   13 u_m    f32  [T][D]   14 c_m bf16 [T][D]  15 al_m f32 [T]
 *   16 acc_up i32  [T][F]   17 g   f32 [T][F]  (GeLU output, quantiser input)
 *   18 c_d    bf16 [T][F]   19 al_d f32 [T]    20 acc_d i32 [T][D]
 *   21 h_out  f32  [T][D]    after the down-projection residual
 * Returns VLA_ERR_INVALID_ARG for a dense handle, a bad step, or a short or
 * misaligned buffer. */
vla_status vla_expert_w2a8_tap_bytes(const vla_expert* h, int B, size_t* bytes);
vla_status vla_expert_set_w2a8_tap(vla_expert* h, int step, void* tap_dev, size_t bytes);

/* Eq. 4, first line, as a standalone op.  Runs the row quantiser the W2A8
 * solver runs on its fp32 rows (the same kernel template; the solver stores
 * the codes as exact bf16 carriers, this entry point as int8):
 *   x_dev     [M][K] fp32 rows
 *   a_dev     [M][K] int8 out: clip(round_half_even(x / alpha_m), -128, 127)
 *   alpha_dev [M] fp32 out: max(|x_m|_inf, 1e-5) / 127 (IEEE division)
 * M >= 1, 1 <= K <= 53248. */
vla_status vla_w2a8_quantize_rows(const float* x_dev, int M, int K, int8_t* a_dev,
                                  float* alpha_dev, void* stream);

/* Eq. 4, second line, as a standalone op:
 *   a_dev      [M][K] int8, alpha_dev [M] fp32
 *   q_dev      [N][K/4] packed ternary codes (as in vla_expert_weights_w2a8)
 *   beta       per-tensor fp32 scale
 *   y_dev      [M][N] bf16 (raw uint16 bits) out: bf16_rne((float(acc) * alpha_m) * beta)
 *   acc_dev    NULL or [M][N] int32 out: acc_mn = sum_j a_mj q_nj (exact)
 * K must be a multiple of 64 with 64 <= K <= 65536 (so every |acc| stays
 * below 2^24 and the fp32 accumulation is exact), and N a multiple of 4.
 * Codes are assumed valid (3 is not checked here).  Runs on the tensor
 * cores: the int8 codes are carried exactly in bf16 and every partial sum is
 * an integer below 2^24, so the fp32 accumulators equal the int32
 * definition.  Allocates its scratch from the stream's memory pool. */
vla_status vla_w2a8_ternary_gemm(const int8_t* a_dev, const float* alpha_dev, const uint8_t* q_dev,
                                 float beta, int M, int N, int K, uint16_t* y_dev,
                                 int32_t* acc_dev, void* stream);

/* Allocation-free variant of vla_w2a8_ternary_gemm.  The paper has no
 * counterpart; it exists for callers that cannot allocate device memory
 * while they run -- a robot control loop with a hard period, where a device
 * allocation may synchronise the device or take an unbounded time, or a host
 * program whose device memory is reserved up front by another runtime's
 * pool.  Same arguments, layouts, limits and results (bit for bit) as
 * vla_w2a8_ternary_gemm, with one more requirement: a_dev must be 4-byte
 * aligned (its kernel reads the codes as 32-bit words; a misaligned a_dev is
 * refused with VLA_ERR_INVALID_ARG before anything is enqueued).  Its fp32
 * partial-sum scratch is a fixed array of VLA_NOALLOC_MAX_ELEMS floats
 * (4 MiB) inside the library, held by every GPU that loads the library until
 * the process exits; the call itself makes no allocation.
 *   - M * N > VLA_NOALLOC_MAX_ELEMS -> VLA_ERR_UNSUPPORTED (nothing enqueued).
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.  The address is cached per device ordinal: after a
 *     cudaDeviceReset of a device, do not call this entry point on it again
 *     in the same process.
 *   - All calls share the array, which keeps the last call's contents; calls
 *     that overlap on the GPU race on it, so order them (one stream, or
 *     explicit dependencies).  Nothing needs clearing between calls: every
 *     call overwrites the M x N slots it reads. */
#define VLA_NOALLOC_MAX_ELEMS 1048576
vla_status vla_w2a8_ternary_gemm_noalloc(const int8_t* a_dev, const float* alpha_dev, const uint8_t* q_dev,
                                         float beta, int M, int N, int K, uint16_t* y_dev,
                                         int32_t* acc_dev, void* stream);

/* Diagnostic: the exact GeLU x Phi(x) of the few-token kernels (erff) and the
 * form the many-token linear epilogue uses (erf by Abramowitz & Stegun 7.1.26,
 * |error| <= 1.5e-7, with approximate reciprocal and exponential), both for
 * n fp32 inputs x_dev into exact_dev and fast_dev. */
vla_status vla_debug_gelu_forms(const float* x_dev, int n, float* exact_dev, float* fast_dev, void* stream);

/* Selected FFN neurons (the rMuscle Action Cache: during the memory-bound
 * denoising loop the expert evaluates only chosen MLP neurons).  idx_dev
 * int32 [L][F_sel]: strictly increasing neuron indices in [0, F) per layer.
 * Builds handle-owned compact copies of the selected rows of W_up and
 * columns of W_down (allocated by the first selection), after which every
 * denoise call on this handle streams only those (MLP width F_sel); F_sel = 0
 * restores the full MLP.  F_sel must be a multiple of 128.  Dense bf16
 * handles on the tensor-core path only (else VLA_ERR_UNSUPPORTED); bad
 * indices -> VLA_ERR_INVALID_ARG with the previous state kept.  Synchronises
 * `stream`; drops the handle's captured graphs. */
vla_status vla_expert_select_ffn(vla_expert* h, const int32_t* idx_dev, int F_sel, void* stream);

/* Number of kernels one denoise call launches for batch B and prefix P
 * (all of them inside the one graph launch).  Host-only arithmetic. */
vla_status vla_expert_launch_count(const vla_expert* h, int B, int P, int* kernels);

/* Human-readable name of a status. */
const char* vla_status_string(vla_status s);

/* Text of the last CUDA failure seen by this thread (the call and the CUDA
 * error), "" if none; valid until the next failing call on this thread. */
const char* vla_last_error(void);

/* Library version, e.g. "0.1.0". */
const char* vla_version(void);

#ifdef __cplusplus
}
#endif
#endif /* VLA_H_ */
