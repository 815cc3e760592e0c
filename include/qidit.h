/*
 * qidit.h - C ABI of the GB300 (sm_103a) Qwen-Image-2.1 DiT step library.
 *
 * The library runs the forward pass of the 7B single-stream DiT denoiser of
 * Qwen-Image-2.1 once per FlowMatch Euler step, plus the host-contract pieces
 * around it (RoPE tables, sigma schedule, noise packing, Euler update).
 *
 * Sources (page titles, sections):
 *   [ARCH]  "Qwen-Image-2.1 Core AI port" (coreai-model-zoo knowledge page),
 *           architecture table, DiT row: 32 single-stream blocks, one shared
 *           modulation Linear 4096->16384 with rows for the sampled t and t = 0,
 *           ZeroCenterRMSNorm text projection, SwiGLU x3, 3-axis interleaved
 *           RoPE (16/56/56), block-causal attention; graph I/O shapes.
 *   [HOST]  "Host contract - RGBA-Image-2.1", section 1 (graph I/O, fp32 at the
 *           boundary), section 4 (sequence layout, positions, RoPE tables),
 *           section 5 (noise packing), section 6 (sampler).
 *   [REUSE] "Qwen-Image-2.1 on MLX, faster and exact", section "Text K/V reuse":
 *           text rows use the t = 0 modulation row and causal attention over
 *           text only, so their K/V are constant over a whole run.
 *
 * Conventions for every call:
 *   - Tensor arguments are DEVICE pointers (memory of the device the handle was
 *     created on) unless the argument says "host".
 *   - Floating-point tensors crossing the boundary are float32, row-major.
 *     Weights are bfloat16 bit patterns (uint16_t), row-major [out, in]. The
 *     library keeps the tensor-core weights as fp16 (converted once at load:
 *     exact for |w| >= 2^-14, error < 2^-25 below; |w| > 65504 is rejected) and
 *     runs every tensor-core product on fp16 operands with fp32 accumulation;
 *     the residual stream, norms and modulation stay fp32.
 *   - Work is enqueued on `stream` (0 = legacy default stream); calls return
 *     without synchronising unless stated. The caller owns every buffer it
 *     passes; the library never keeps a caller pointer after a call returns.
 *   - Errors are returned, never thrown; qi_last_error() gives the calling
 *     thread's last message. Device-side wait timeouts (which are bugs, not
 *     expected events) are latched in a device error word and reported by
 *     qi_dit_check() and by the next qi_dit_* call that synchronises.
 *   - Calls on one qi_dit handle must not overlap across streams or threads.
 */
#ifndef QIDIT_H
#define QIDIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qi_stream_t; /* same handle as cudaStream_t */

typedef enum qi_status {
  QI_OK = 0,
  QI_ERR_INVALID_ARG = 1,     /* NULL pointer, bad enum, bad block index        */
  QI_ERR_SHAPE = 2,           /* L, N, h, w out of range or over the handle's max */
  QI_ERR_STATE = 3,           /* e.g. USE_CACHE with no valid capture for this L */
  QI_ERR_OOM = 4,             /* device allocation failed                       */
  QI_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed              */
  QI_ERR_DEVICE_TIMEOUT = 6,  /* a kernel's bounded wait expired (device word)  */
  QI_ERR_NOT_IMPLEMENTED = 7,
  QI_ERR_NONFINITE = 8        /* a pass produced a non-finite velocity (device word) */
} qi_status;

/* Model widths [ARCH]. head_dim 128 follows from the 64 RoPE columns per token
 * (one column per rotated pair); SwiGLU width 12288 = 3 x 4096. */
#define QI_HIDDEN 4096
#define QI_HEADS 32
#define QI_HEAD_DIM 128
#define QI_FFN 12288
#define QI_MOD (4 * QI_HIDDEN) /* (s1, g1, s2, g2) */
#define QI_PATCH 64            /* latent channels per image token */
#define QI_TDIM 256            /* sinusoidal timestep width       */
#define QI_BLOCKS 32
#define QI_ROPE_COLS 64        /* 8 + 28 + 28 pairs per token     */
#define QI_ROPE_POS_LO (-1024)
#define QI_ROPE_NPOS 9216      /* positions -1024..8191           */

/* Accepted sizes. L is the prompt length after the template prefix is dropped
 * [HOST s2]; N = h*w image tokens. The pages' N axis stops at 4096 but their
 * 2048^2 default is 16384 tokens, so N goes to 16384 here. */
#define QI_L_MIN 1
#define QI_L_MAX 512
#define QI_N_MIN 1
#define QI_N_MAX 16384

/* qi_dit_step flags */
#define QI_STEP_JOINT 0u      /* text + image rows; (re)captures the text K/V       */
#define QI_STEP_USE_CACHE 1u  /* image rows only; text K/V come from the capture    */
#define QI_STEP_HOST_IO 2u    /* img_tokens, txt_feats, cos/sin, vel are HOST ptrs  */

typedef struct qi_dit qi_dit;

typedef struct qi_dit_config {
  int blocks; /* 1..32 (32 for the real model; fewer for tests)                 */
  int L_max;  /* largest prompt length this handle serves (1..512)              */
  int N_max;  /* largest image token count this handle serves (1..16384)        */
  int kv_slots; /* text K/V slots: 0 or 1 = one; 2 = a second slot for the negative
                 * prompt of classifier-free guidance (qi_dit_step_cfg)          */
  int mxfp8;    /* 1 = also keep MXFP8 copies of the block weights (+7.1 GB at 32
                 * blocks) so that passes can run on block-scaled GEMMs
                 * (qi_dit_set_mxfp8); 0 = fp16 only                             */
} qi_dit_config;

/* Global (non-block) tensors, bf16 bits, [out, in] row-major. */
typedef struct qi_global_weights {
  const uint16_t* t_w1;       /* [4096, 256]  timestep MLP, first Linear        */
  const uint16_t* t_b1;       /* [4096]                                        */
  const uint16_t* t_w2;       /* [4096, 4096] timestep MLP, second Linear       */
  const uint16_t* t_b2;       /* [4096]                                        */
  const uint16_t* mod_w;      /* [16384, 4096] the one shared modulation Linear */
  const uint16_t* mod_b;      /* [16384]                                       */
  const uint16_t* txt_norm_w; /* [4096] ZeroCenterRMSNorm gain w (scale 1 + w)  */
  const uint16_t* txt_w;      /* [4096, 4096] text projection                   */
  const uint16_t* txt_b;      /* [4096]                                        */
  const uint16_t* img_w;      /* [4096, 64] image-token projection              */
  const uint16_t* img_b;      /* [4096]                                        */
  const uint16_t* out_w;      /* [64, 4096] proj_out                            */
  const uint16_t* out_b;      /* [64]                                          */
} qi_global_weights;

/* One block's matrices, bf16 bits, [out, in] row-major. No biases. */
typedef struct qi_block_weights {
  const uint16_t* wq; /* [4096, 4096]  */
  const uint16_t* wk; /* [4096, 4096]  */
  const uint16_t* wv; /* [4096, 4096]  */
  const uint16_t* wo; /* [4096, 4096]  */
  const uint16_t* wg; /* [12288, 4096] SwiGLU gate */
  const uint16_t* wu; /* [12288, 4096] SwiGLU up   */
  const uint16_t* wd; /* [4096, 12288] SwiGLU down */
} qi_block_weights;

/* Sampler constants [HOST s6, scheduler.json]. */
typedef struct qi_sched_params {
  double base_shift;     /* 0.5  */
  double max_shift;      /* 0.9  */
  int base_seq;          /* 256  */
  int max_seq;           /* 8192 */
  double shift_terminal; /* 0.02 */
  int train_steps;       /* 1000 */
} qi_sched_params;

/* ------------------------------------------------------------------ lifetime */

/* Create a handle on CUDA device `device`: allocates the bf16 weight store
 * (~14.2 GB at 32 blocks), activations for L_max + N_max rows and the per-block
 * text K/V store. Weights start undefined: load them with qi_dit_load_*.
 * Errors: INVALID_ARG (NULL), SHAPE (config out of range), OOM, CUDA. */
qi_status qi_dit_create(const qi_dit_config* cfg, int device, qi_dit** out);

/* Free everything the handle owns. Synchronises the device. NULL is a no-op. */
qi_status qi_dit_destroy(qi_dit* dit);

/* Copy the global tensors into the handle. `src_on_device` = 1 when the
 * pointers are device memory, 0 when host memory. Returns after the copies
 * completed, so the caller may free its copy. */
qi_status qi_dit_load_global(qi_dit* dit, const qi_global_weights* w, int src_on_device,
                             qi_stream_t stream);

/* Copy block `block`'s matrices into the handle (repacked internally: Q|K|V
 * stacked, gate/up interleaved by 64-row groups). Returns after completion. */
qi_status qi_dit_load_block(qi_dit* dit, int block, const qi_block_weights* w,
                            int src_on_device, qi_stream_t stream);

/* ------------------------------------------------------------------ host contract */

/* The three RoPE axis tables [HOST s4]: for axis widths d = 16, 56, 56 and
 * positions p = -1024..8191 (row p + 1024), column k < d/2 holds
 * cos/sin(fl32(fl32(p) * omega_k)), omega_k = fl32(theta^(-2k/d)); each value
 * is the float32 rounding of the float64 cos/sin. Outputs (device, float32):
 * cos0/sin0 [9216, 8], cos1/sin1 [9216, 28], cos2/sin2 [9216, 28]. */
qi_status qi_rope_axis_tables(float theta, float* cos0, float* sin0, float* cos1, float* sin1,
                              float* cos2, float* sin2, qi_stream_t stream);

/* Per-token RoPE rows [HOST s4]: text token i has position (i, i, i); image
 * token y*w + x has (L, y - (h - h/2), x - (w - w/2)); a token's 64 columns are
 * the axis-0, axis-1, axis-2 rows concatenated (8 + 28 + 28), same values as
 * qi_rope_axis_tables. Outputs (device, float32): txt_cos/txt_sin [L, 64],
 * img_cos/img_sin [h*w, 64]. Any of the four may be NULL (skipped).
 * Errors: SHAPE if L or h*w is out of range. */
qi_status qi_rope_tables(int L, int h, int w, float theta, float* txt_cos, float* txt_sin,
                         float* img_cos, float* img_sin, qi_stream_t stream);

/* FlowMatch Euler schedule [HOST s6], computed on the host:
 * s = linspace(1, 1/steps, steps); mu = N*m + b (m, b from the constants);
 * s = e^mu / (e^mu + 1/s - 1); s = 1 - (1 - s) / ((1 - s_last) / (1 - shift_terminal));
 * evaluated in float64, then timesteps[i] = fl32(s_i * train_steps) and
 * sigmas = fl32(s) ++ [0]. `p` may be NULL (the constants above).
 * Outputs (HOST): sigmas [steps + 1], timesteps [steps]. The DiT's timestep input
 * for step i is fl32(timesteps[i] / 1000). Errors: INVALID_ARG, SHAPE (steps < 2: with a
 * single step its only sigma is 1 and the terminal stretch divides 0 by 0). */
qi_status qi_flow_sigmas(int steps, int N, const qi_sched_params* p, float* sigmas,
                         float* timesteps);

/* Noise packing [HOST s5]: x[y*w + x, c] = z[c, y, x] for a channel-major
 * latent z [64, h, w] (device) into tokens x [h*w, 64] (device). */
qi_status qi_pack_noise(const float* z, int h, int w, float* x, qi_stream_t stream);

/* Euler update [HOST s6]: x <- x + (sigma_next - sigma_i) * vel, float32, the
 * difference, the product and the sum each rounded on its own (no FMA).
 * x, vel: device [N, 64]. */
qi_status qi_euler_update(float* x, const float* vel, int N, float sigma_i, float sigma_next,
                          qi_stream_t stream);

/* DPM++ 2M sampler [MLX page, "Optional modes (approximate or slower)": offered
 * next to Euler, no formula given]. Reading: the multistep second-order
 * DPM-Solver++ (Lu et al. 2022) on the flow-matching schedule alpha = 1 - sigma,
 * lambda = log(alpha / sigma), with the data prediction D = x - sigma * vel.
 * Step i (sigma_i -> sigma_{i+1}), a = sigma_{i+1} / sigma_i, b = 1 - a:
 *   order 2:  x <- a x + b (c0 D - c1 D_prev),  c1 = h_i / (2 h_{i-1}), c0 = 1 + c1,
 *             h_i = lambda_{i+1} - lambda_i;
 *   order 1:  x <- a x + b D   (i = 0, or sigma_{i-1} = 1 where lambda = -inf);
 *   order 0:  x <- D           (sigma_{i+1} = 0, the last step).
 *
 * qi_dpmpp2m_coeffs (host only, no device work): the step's order and
 * coefficients {a, b, c0, c1}, each evaluated in float64 from the float32 sigmas
 * and rounded once to float32. sigmas: HOST [steps + 1]; coeffs: HOST [4].
 * Errors: INVALID_ARG (NULL, i outside 0..steps-1, sigmas not decreasing from
 * <= 1 to >= 0 over steps i-1..i+1), SHAPE (steps < 1).
 *
 * qi_dpmpp2m_update: applies step i in float32, every operation rounded on its
 * own (no FMA): D = x - fl(sigma_i vel); order 2: D' = fl(c0 D) - fl(c1 D_prev);
 * x = fl(a x) + fl(b D'). Then d_prev <- D for step i + 1. x, vel, d_prev:
 * device [N, 64] float32; d_prev is read only by second-order steps (its
 * contents may be anything before step 0). sigmas: HOST [steps + 1]. */
qi_status qi_dpmpp2m_coeffs(const float* sigmas, int steps, int i, int* order, float* coeffs);
qi_status qi_dpmpp2m_update(float* x, const float* vel, float* d_prev, int N, const float* sigmas,
                            int steps, int i, qi_stream_t stream);

/* ------------------------------------------------------------------ DiT */

/* One DiT forward pass [ARCH; HOST s1]: vel [N, 64] from img_tokens [N, 64],
 * txt_feats [L, 4096], the scalar timestep (t = timesteps[i] / 1000) and the
 * per-token RoPE rows txt_cos/txt_sin [L, 64], img_cos/img_sin [N, 64].
 *
 * flags = QI_STEP_JOINT: all L + N rows run through every block; the text K/V
 *   of every block are stored in the handle (the capture), valid for this L.
 * flags = QI_STEP_USE_CACHE [REUSE]: only the N image rows run; attention reads
 *   the stored text K/V. txt_feats and txt_cos/txt_sin may be NULL. The result
 *   equals the joint pass's image rows bit for bit (every GEMM computes a row
 *   independently of the others, and attention walks keys in the same order).
 *   Errors: STATE if no capture is valid for this L.
 * | QI_STEP_HOST_IO: the tensor pointers are host memory; the library copies
 *   them in and vel out on `stream`, and synchronises it before returning.
 * Errors: INVALID_ARG, SHAPE (L > L_max, N > N_max, ...), STATE, CUDA. */
qi_status qi_dit_step(qi_dit* dit, const float* img_tokens, int N, const float* txt_feats, int L,
                      float timestep, const float* txt_cos, const float* txt_sin,
                      const float* img_cos, const float* img_sin, float* vel, unsigned flags,
                      qi_stream_t stream);

/* One FlowMatch Euler sampler step [HOST s6; ARCH]: the DiT pass of qi_dit_step
 * with x (the latent tokens [N, 64], float32) as img_tokens, then the Euler update
 * of qi_euler_update in place, x <- x + (sigma_next - sigma_i) * vel (each
 * operation rounded on its own), so one call advances the sampler by one step.
 * Arguments and flags as qi_dit_step; timestep is the DiT input of the step
 * (timesteps[i] / 1000), sigma_i and sigma_next its two sigmas. vel_out [N, 64]
 * receives the velocity; it may be NULL, and then the velocity stays in the
 * handle's staging buffer. With QI_STEP_HOST_IO, x (in and out), txt_feats, the
 * four tables and vel_out are HOST pointers (pinned memory copies fastest): the
 * call copies the inputs in, x (and vel_out) out, and synchronises `stream`
 * before returning, reporting a device-word error as qi_dit_check does.
 * The first call with host buffers or a NULL vel_out allocates the staging
 * buffers (inputs and velocity for N_max and L_max rows, held until destroy).
 * x, vel_out: element-wise identical to qi_dit_step followed by qi_euler_update.
 * Errors: as qi_dit_step; INVALID_ARG for non-finite sigmas; OOM for staging. */
qi_status qi_dit_euler_step(qi_dit* dit, float* x, int N, const float* txt_feats, int L, float timestep,
                            float sigma_i, float sigma_next, const float* txt_cos, const float* txt_sin,
                            const float* img_cos, const float* img_sin, float* vel_out, unsigned flags,
                            qi_stream_t stream);

/* Classifier-free guidance step [MLX page, "Optional modes": the negative
 * prompt is used as noise = neg + g * (pos - neg), with its K/V in a second
 * slot ("Text K/V reuse")]. Runs the pass of qi_dit_step for the conditional
 * prompt (K/V slot 0) and for the negative prompt (slot 1) on the same
 * img_tokens and timestep, then vel = neg + guidance * (pos - neg) in float32,
 * each operation rounded on its own. Each prompt has its own tables: image
 * positions carry the prompt length in their frame coordinate.
 * flags = QI_STEP_JOINT: both passes are joint and capture their slot.
 * flags = QI_STEP_USE_CACHE: image rows only, both prompts in ONE pass of 2N
 * rows (batch 2: every GEMM runs once on both prompts' rows; attention runs per
 * prompt over its own K/V); each half equals that prompt's own image-only pass
 * bit for bit. The *_feats and *_txt_* tensors may be NULL; the captures must be
 * for L_pos and L_neg.
 * Errors: STATE (handle created with kv_slots != 2, no matching capture),
 * SHAPE, INVALID_ARG, CUDA. */
qi_status qi_dit_step_cfg(qi_dit* dit, const float* img_tokens, int N, float timestep, float guidance,
                          const float* pos_feats, int L_pos, const float* pos_txt_cos, const float* pos_txt_sin,
                          const float* pos_img_cos, const float* pos_img_sin, const float* neg_feats, int L_neg,
                          const float* neg_txt_cos, const float* neg_txt_sin, const float* neg_img_cos,
                          const float* neg_img_sin, float* vel, unsigned flags, qi_stream_t stream);

/* First-block cache, "Fast mode" [MLX page, "Optional modes (approximate or
 * slower)": block 0 always runs; blocks 1 to 31 are skipped while block 0's
 * residual changes less than a threshold; options table: 0.08]. Approximate.
 *
 * One qi_dit_step (same arguments and flags, QI_STEP_HOST_IO excepted) under the
 * cache. Block 0 runs on every row; r0 = x1 - x0 on the image rows (x0 entering
 * block 0, x1 leaving it) is compared with the reference r0_ref of the last call
 * that ran every block: rel = sum |r0 - r0_ref| / sum |r0_ref| (fp32 terms, fp64
 * sums). If rel < threshold the call skips blocks 1..last and the head reads
 * x1 + rest, where rest = x_last - x1 of the reference call; otherwise it runs
 * every block and becomes the new reference (r0_ref, rest). There is no
 * reference after qi_dit_fbcache_reset, a joint pass (any entry point), a text
 * capture, or a change of N or L; such a call runs every block (rel = +inf).
 *
 * threshold: skip when rel < threshold (0 never skips). rel_change, skipped: HOST
 * outputs (may be NULL): the measure (+inf without a reference) and 1 if blocks
 * were skipped. With a reference the call synchronises `stream` to read the
 * measure. The first call allocates 5 x N_max x 4096 float32 of device memory
 * for the cache (held until qi_dit_destroy).
 * Errors: as qi_dit_step; INVALID_ARG for QI_STEP_HOST_IO or a NaN threshold. */
qi_status qi_dit_step_fbcache(qi_dit* dit, const float* img_tokens, int N, const float* txt_feats,
                              int L, float timestep, const float* txt_cos, const float* txt_sin,
                              const float* img_cos, const float* img_sin, float threshold,
                              float* vel, float* rel_change, int* skipped, unsigned flags,
                              qi_stream_t stream);

/* Drops the first-block cache's reference: the next qi_dit_step_fbcache runs every
 * block. Host only. Errors: INVALID_ARG (NULL). */
qi_status qi_dit_fbcache_reset(qi_dit* dit);

/* Text-only pass [REUSE]: run the L text rows (t = 0 modulation, causal over
 * text) through every block and store their K/V, the same values a joint pass
 * stores. No velocity. Marks the capture valid for this L. */
qi_status qi_text_kv_capture(qi_dit* dit, const float* txt_feats, int L, const float* txt_cos,
                             const float* txt_sin, qi_stream_t stream);

/* Bytes of text K/V storage for `blocks` blocks and L tokens [REUSE]:
 * 2 x blocks x L x 4096 x 2. */
size_t qi_kv_cache_bytes(int blocks, int L);

/* Device error word: synchronises `stream`; returns DEVICE_TIMEOUT if a kernel's
 * bounded wait expired, or NONFINITE if a pass produced a non-finite velocity,
 * since the last check (and clears the word). */
qi_status qi_dit_check(qi_dit* dit, qi_stream_t stream);

/* ------------------------------------------------------------------ test hooks */

/* One block in the joint layout: hidden [L + N, 4096] float32 in/out (text rows
 * first), modulation rows for t_img (image rows) and 0 (text rows), per-row
 * RoPE cos/sin [L + N, 64]. Stores the block's K/V like a joint step. */
qi_status qi_dit_block_forward(qi_dit* dit, int block, float* hidden, int L, int N, float t_img,
                               const float* cos, const float* sin, qi_stream_t stream);

/* Copy rows [row0, row0 + rows) of block `block`'s stored K and V (fp16 bits,
 * [rows, 4096] each, device) into k_out / v_out. After a pass, rows [0, L) are
 * the text K/V (post-RoPE K) and rows [L, L + N) the image K/V of that pass.
 * Errors: INVALID_ARG (block, NULL), SHAPE (rows past L_max + N_max). */
qi_status qi_dit_read_kv(qi_dit* dit, int block, int row0, int rows, uint16_t* k_out, uint16_t* v_out,
                         qi_stream_t stream);

/* The block's tensor-core GEMM on its own, plain fp32 output (test hook):
 * D[M, N] = A[M, K] * B[N, K]^T with A, B bf16 bits row-major (device).
 * Requires N % 256 == 0, K % 64 == 0, 16-byte aligned A and B; M >= 1 any.
 * Uses the handle's device error word. Errors: SHAPE, INVALID_ARG, CUDA. */
qi_status qi_gemm_bf16(qi_dit* dit, const uint16_t* A, const uint16_t* B, float* D, int M, int N, int K,
                       qi_stream_t stream);

/* Failure injection for tests [failure detection: every device wait is bounded].
 * The pages have no counterpart; it lets a test see the library's error paths
 * without faulting, trapping or hanging the GPU.
 * kind 1: the arg-th next device allocation made by the library (process-wide,
 *   dit may be NULL) fails as if the device were out of memory: the call that
 *   makes it returns QI_ERR_OOM and frees what it had allocated.
 * kind 2: the next block GEMM launched for `dit` first waits on a barrier that
 *   nothing arrives on; after the 2 s limit the launch records a timeout in the
 *   device error word and winds down (its copies drained, tensor memory freed).
 *   The pass's result is then undefined; qi_dit_check (or the next call that
 *   synchronises) returns QI_ERR_DEVICE_TIMEOUT and clears the word, and later
 *   calls run normally.
 * kind 0: cancel pending injections (of `dit`, if given).
 * Errors: INVALID_ARG (unknown kind, arg < 1 for kind 1, NULL dit for kind 2). */
qi_status qi_debug_inject(qi_dit* dit, int kind, int arg);

/* ------------------------------------------------------------------ MXFP8 */

/* Block-scaled low-precision GEMMs [MLX page: 4-bit quantised weights, an int8
 * "per_block 32" experiment; Core AI page: int8 / 4-bit weight quantisation].
 * GB300 reading: OCP MX v1.0 MXFP8, i.e. blocks of 32 consecutive values along
 * the contraction axis share one scale 2^e (UE8M0 byte e + 127) and each value
 * is FP8 E4M3; e = floor(log2 max|v|) - 8 clamped to [-127, 127] (-127 for an
 * all-zero block), v * 2^-e rounded to nearest even and clamped to +-448.
 *
 * qi_dit_set_mxfp8: on = 1 runs the four block GEMMs of every later pass (QKV,
 * out-projection, gate/up, down) on MXFP8 weights (quantised from the bf16
 * values at load) and MXFP8 activations (quantised from the fp16 operands just
 * before each GEMM); the pre-norm GEMMs quantise x * (1 + s) and scale the product
 * by the row's 1/rms. on = 0 returns to fp16. Switching drops the text K/V
 * captures and the first-block cache's reference. Host only.
 * Errors: INVALID_ARG (NULL), STATE (handle created with mxfp8 = 0). */
qi_status qi_dit_set_mxfp8(qi_dit* dit, int on);

/* MXFP8 quantisation along K of a row-major [rows, K] 16-bit matrix (bf16 bits
 * if in_is_bf16, else fp16; device, 16-byte aligned): q [rows, K] E4M3 bytes
 * (device, 16-byte aligned) and sf, the scales in 512-byte chunks, chunk
 * (K-group k / 128, row group r / 128) at ((k / 128) * ceil(rows / 128) + r / 128) * 512,
 * byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (k / 32) % 4 within it; sf holds
 * ceil(rows / 128) * (K / 128) * 512 bytes (bytes of rows past `rows` are left
 * as they were). Errors: INVALID_ARG, SHAPE (K % 128 != 0). */
qi_status qi_quant_mxfp8(const uint16_t* in, int in_is_bf16, int rows, int K, uint8_t* q, uint8_t* sf,
                         qi_stream_t stream);

/* The block-scaled GEMM on its own (test hook): D[M, N] = A[M, K] * B[N, K]^T,
 * fp32 out, with A, B and their scales as qi_quant_mxfp8 writes them (device).
 * Requires N % 256 == 0, K % 128 == 0. Uses the handle's device error word.
 * Errors: SHAPE, INVALID_ARG, CUDA. */
qi_status qi_gemm_mxfp8(qi_dit* dit, const uint8_t* A, const uint8_t* A_sf, const uint8_t* B,
                        const uint8_t* B_sf, float* D, int M, int N, int K, qi_stream_t stream);

/* qi_gemm_bf16 without a handle and without allocating. The pages have no
 * counterpart: this exists for callers that may not call the CUDA allocator,
 * such as code inside a host that owns all device memory (an inference server
 * with a fixed arena, a plugin barred from cudaMalloc); they cannot create a
 * qi_dit handle, whose creation allocates the weight store and work buffers.
 * Same kernel, same result as qi_gemm_bf16: D[M, N] = A[M, K] * B[N, K]^T,
 * bf16 bits in, fp32 out, all device pointers owned by the caller.
 * Scratch: the kernel's status word sits in a 256-byte static device array
 * that the library holds on every device that loads it, until exit. The first
 * call on a device (the device current at the call) looks the array up with
 * cudaGetSymbolAddress; make that first call before any stream capture. The
 * address is kept for the life of the process: do not use this entry point on
 * a device after cudaDeviceReset (or another teardown of its primary context).
 * Every call clears the status word, then the kernel reports into it, so calls
 * that overlap on the GPU (other streams, other threads) race on it; serialise
 * them. Limits: N % 256 == 0, K % 64 == 0, M <= 32768, N <= 24576, K <= 12288
 * (the DiT's own GEMM shapes: rows of a joint pass, L + N <= 16896, or of the
 * batch-2 guidance pass, 2 N <= 32768); larger sizes return QI_ERR_SHAPE with a
 * message in qi_last_error(). sync_check != 0 synchronises `stream` and returns
 * QI_ERR_DEVICE_TIMEOUT if a bounded wait in the kernel expired. */
qi_status qi_gemm_bf16_noalloc(const uint16_t* A, const uint16_t* B, float* D, int M, int N, int K,
                               int sync_check, qi_stream_t stream);

/* The block-causal attention kernel on its own (test hook). q [Rq, 4096],
 * k/v [Lk, 4096], o [Rq, 4096], fp16 bits, 32 heads x 128 (device). Query row
 * r has global index r + q_off: if that is < L it sees keys 0..index (text,
 * causal), otherwise keys 0..Lk-1. Scale 1/sqrt(128). */
qi_status qi_attention_f16(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, int Rq,
                            int q_off, int L, int Lk, qi_stream_t stream);

/* The two-row GEMV of the timestep MLP and the shared modulation on its own (test
 * hook; Core AI page, architecture table: the modulation Linear 4096 -> 16384
 * shared by all blocks, with a row for the sampled t and a row for t = 0):
 * y[r][o] = W[o] . act(x[r]) + b[o] for r = 0, 1, act = SiLU if silu_in else the
 * identity. x float32 [2, in_dim], W bf16 bits [out_dim, in_dim] row-major, b bf16
 * bits [out_dim], y float32 [2, out_dim], all device; in_dim is 256 or 4096
 * (else QI_ERR_SHAPE), x and W 16-byte aligned when in_dim = 4096. The caller owns
 * every buffer; the call only enqueues on `stream`. */
qi_status qi_gemv_bf16(const float* x, int in_dim, const uint16_t* W, const uint16_t* b, int out_dim, float* y,
                       int silu_in, qi_stream_t stream);

/* During later qi_dit_step calls, copy the float32 residual stream entering
 * block `block` ([R, 4096], R = rows of that pass; `block` = blocks means the
 * stream after the last block) into `dst` (device). slot 0 or 1; dst NULL clears. */
qi_status qi_dit_set_trace(qi_dit* dit, int slot, int block, float* dst);

/* fp16 operand ranges (test hook). The tensor-core operands are fp16, whose
 * largest finite value is 65504; this records how close a pass comes to it.
 * While `out` is set (device float32 [blocks][QI_RANGE_KINDS], filled with zeros
 * by the caller), every later single-prompt pass of the fp16 mode folds, per
 * block, the largest |value| of each fp16 operand it writes into out with an
 * atomic max (a NaN counts as +inf). Kinds: 0 x (1 + s1), the Q/K/V GEMM's input;
 * 1 Q after RoPE; 2 K after RoPE (the pass's rows of the block's K store); 3 V;
 * 4 the attention output O; 5 x (1 + s2), the gate/up GEMM's input; 6 h, the
 * SwiGLU output and down GEMM input; 7 the text projection's input (in block 0's
 * row only). One extra reduction launch per operand; NULL turns it off.
 * Errors: INVALID_ARG (NULL handle, misaligned out). */
#define QI_RANGE_KINDS 8
qi_status qi_dit_set_range_probe(qi_dit* dit, float* out);

/* Per-kernel-class device time, measured with CUDA events on the launching
 * stream while enabled. Classes: 0 QKV GEMM, 1 attention, 2 out-proj GEMM,
 * 3 gate/up GEMM, 4 down GEMM, 5 other. Each timed launch group adds two event
 * records to the stream, and an event between two kernels also stops the second
 * from starting its set-up under the first, so timing every class slows a pass
 * by roughly 1 %. qi_dit_profile: enable != 0 times every class in every block,
 * 0 none. qi_dit_profile_classes: times only the classes whose bit (1 << class)
 * is set in `mask` (0 = none), and the per-block classes 0-4 only in blocks b
 * with b % block_stride == 0 (1 = every block). Bits at or above
 * QI_PROF_CLASSES or block_stride < 1 give QI_ERR_INVALID_ARG. Either call
 * resets the counters. */
#define QI_PROF_CLASSES 6
qi_status qi_dit_profile(qi_dit* dit, int enable);
qi_status qi_dit_profile_classes(qi_dit* dit, unsigned mask, int block_stride);
/* Synchronises; writes total milliseconds and launch counts per class since
 * the last reset, then resets. ms/launches: host arrays [QI_PROF_CLASSES]. */
qi_status qi_dit_profile_read(qi_dit* dit, double* ms, long long* launches);

/* Message for the calling thread's last failed call ("" if none). */
const char* qi_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* QIDIT_H */
