/*
 * mi_block: forward pass of a MOSS-Image-style diffusion-transformer (DiT) block on one GB300
 * (sm_103a), plus one guided denoising step built from it.
 *
 * What the block computes is named on the TensorFold page "MOSS-Image transformer on CUDA"
 * (PR #1528): section "What it adds" lists the hand-written kernels (modulated RMSNorm, q/k norm
 * and rotary into packed rows, the SiLU gate, gated add), the bf16 projections with fp32 sums and
 * the full head-128 attention; its precision bullet fixes bf16 weights and activations with fp32
 * sums, norms and softmax.  The guided step (empty negative prompt, guidance, Euler schedule) is
 * the host loop of PR #2281, section "What this changes".  Where the pages name an operation
 * without its formula, the plain definition is used:
 *
 *   h   = x * rsqrt(mean(x^2) + eps) * (1 + scale1) + shift1
 *   qkv = h W_qkv^T;  q, k per head: RMSNorm over 128 with gain, then rotary on pairs (2p, 2p+1)
 *   o   = softmax(q k^T / sqrt(128) with masked keys at -inf) v
 *   x1  = x + gate1 * (o W_o^T)
 *   h2  = x1 * rsqrt(mean(x1^2) + eps) * (1 + scale2) + shift2
 *   m   = silu(h2 Wg^T) * (h2 Wu^T),  W_gu = [Wg; Wu]
 *   y   = x1 + gate2 * (m W_d^T)
 *
 * Conventions of every entry point:
 *   - All tensors are device pointers owned by the caller; every bf16 tensor is row-major,
 *     16-byte aligned, and passed as `void*` holding __nv_bfloat16 values.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is only enqueued:
 *     nothing here synchronises, allocates device memory on the forward path, prints or aborts.
 *   - Every function returns mi_status; on failure mi_last_error() (thread-local) says why and
 *     nothing was enqueued.
 *   - Results are deterministic: the same inputs on the same GPU and build give the same bytes.
 */
#ifndef MI_BLOCK_H
#define MI_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MI_ABI_VERSION 1

typedef enum mi_status {
  MI_OK = 0,
  MI_ERR_INVALID_ARG = 1,  /* null pointer, misaligned pointer, bad geometry */
  MI_ERR_UNSUPPORTED = 2,  /* device is not sm_103, head_dim != 128, or a shape the kernels refuse */
  MI_ERR_WORKSPACE = 3,    /* workspace pointer null/misaligned or smaller than the query says */
  MI_ERR_CUDA = 4,         /* a CUDA runtime call failed (message carries the CUDA error string) */
  MI_ERR_DEVICE = 5        /* a kernel reported a pipeline timeout through the device error flag */
} mi_status;

/* Thread-local message of the last failed call on this thread ("" if none). */
const char* mi_last_error(void);

/* MI_ABI_VERSION of the loaded library. */
int mi_abi_version(void);

/* MI_OK if the current device is an sm_103 GPU the kernels were built for. */
mi_status mi_device_supported(void);

/* Reads and clears the device error flag of the current device.  *code = 0 when every kernel
 * since the last call finished its pipeline; otherwise the first timeout code recorded (a kernel
 * whose wait ran out of polls, about 1.5 s, returns early and leaves its outputs undefined).
 * Synchronises the device (diagnostic call, not for the hot path). */
mi_status mi_device_error(int* code);

/* Error codes mi_device_error reports: 0x100 + k (a GEMM wait), 0x200 + k (an attention wait),
 * 0x300 (the self-test below), 0x400 (a GEMM whose split of tail tiles over the CTAs has more parts
 * per tile than its fix-up adds; the library's own plans never produce one), 0x500 + k (a wait of
 * the modulated RMSNorm for its row copies). */
#define MI_DEV_TIMEOUT_GEMM 0x100
#define MI_DEV_TIMEOUT_ATTN 0x200
#define MI_DEV_TIMEOUT_SELFTEST 0x300
#define MI_DEV_SCHEDULE_GEMM 0x400
#define MI_DEV_TIMEOUT_NORM 0x500

/* Enqueues a one-CTA kernel whose pipeline wait can never complete: the wait gives up after about
 * limit_us microseconds (at most 1e6; the pipelines' own bounded wait, given as many polls as take
 * that long), records MI_DEV_TIMEOUT_SELFTEST in the device error flag and the kernel returns.
 * Exercises the failure path of the bounded waits without a fault or hang. */
mi_status mi_selftest_wait_timeout(int limit_us, void* stream);

/* ---------------------------------------------------------------------------------- block --- */

typedef struct mi_block_desc {
  int hidden;      /* H: multiple of 256, at most 4096; H = n_heads * head_dim */
  int n_heads;
  int head_dim;    /* must be 128 */
  int mlp_inter;   /* I: multiple of 128 */
  float eps;       /* RMSNorm epsilon of all three norms (1e-6 in the synthetic workloads) */
  int fuse_epilogues; /* 1: SiLU gate fused into the gate/up GEMM and the gated residual adds into
                         the W_o / W_d GEMMs; 0: separate kernels.  Both give identical bytes. */
  /* Weights (bf16, device, read-only, must outlive the mi_block): */
  const void* w_qkv;    /* [3H, H]: rows [0,H) q, [H,2H) k, [2H,3H) v; head j = rows 128j.. of each */
  const void* w_o;      /* [H, H] */
  const void* w_gu;     /* [2I, H]: rows [0,I) gate, [I,2I) up */
  const void* w_d;      /* [H, I] */
  const void* q_norm_w; /* [128]: gain of the per-head q RMSNorm, shared by all heads */
  const void* k_norm_w; /* [128] */
} mi_block_desc;

/* Sequence layout of one batch element: text_pad prompt rows, then grid_h * grid_w image tokens
 * in row-major (r, c) order.  S = text_pad + grid_h * grid_w rows per element. */
typedef struct mi_seq_layout {
  int batch;
  int text_pad;
  int grid_h;
  int grid_w;
} mi_seq_layout;

typedef struct mi_block mi_block;

/* Validates the geometry, the weight pointers and the device (sm_103 required, else
 * MI_ERR_UNSUPPORTED) and builds the TMA descriptors of the weights.  Refuses any null weight.
 * PR #1528, "What it adds": the model's load takes the released geometry only, refuses a tensor
 * it does not read, and refuses GPUs it was not built for (there sm_120/121, here sm_103).
 * The weights stay owned by the caller; *out is released with mi_block_destroy. */
mi_status mi_block_init(mi_block** out, const mi_block_desc* desc);
void mi_block_destroy(mi_block* blk);

/* Workspace bytes mi_block_forward needs for `batch` elements of `seq` rows: one slab per
 * intermediate (h, qkv, packed q/k, o, x1, h2, m, plus a and gu/dn when epilogues are not fused)
 * and the GEMM's stream-K scratch when a projection's plan uses it.  PR #1528, "Measured": the
 * scratch of a forward is computed from its allocations (0.51 GB there at 1024x1024 with a 34-row
 * prompt).  Host arithmetic only. */
mi_status mi_block_workspace_size(const mi_block* blk, int batch, int seq, size_t* bytes);

/* Intermediates left in the workspace by the last forward (for parity checks). */
typedef enum mi_tensor {
  MI_T_H = 0,   /* [B*S, H]  modulated RMSNorm #1 */
  MI_T_QKV = 1, /* [B*S, 3H] QKV projection (with fused epilogues only the v columns [2H, 3H)) */
  MI_T_QP = 2,  /* [B, heads, S, 128] q after norm + rotary */
  MI_T_KP = 3,  /* [B, heads, S, 128] k after norm + rotary */
  MI_T_O = 4,   /* [B*S, H]  attention output, heads concatenated */
  MI_T_A = 5,   /* [B*S, H]  o W_o^T               (only when epilogues are not fused) */
  MI_T_X1 = 6,  /* [B*S, H]  first residual */
  MI_T_H2 = 7,  /* [B*S, H]  modulated RMSNorm #2 */
  MI_T_GU = 8,  /* [B*S, 2I] gate/up projection    (only when epilogues are not fused) */
  MI_T_M = 9,   /* [B*S, I]  SiLU gate */
  MI_T_DN = 10  /* [B*S, H]  down projection       (only when epilogues are not fused) */
} mi_tensor;

/* Byte offset and size of intermediate `which` inside the workspace; MI_ERR_UNSUPPORTED when the
 * block's fusion setting does not materialise it. */
mi_status mi_block_tensor_offset(const mi_block* blk, int batch, int seq, int which, size_t* offset,
                                 size_t* bytes);

/*
 * One block forward over L->batch elements: the seven formulas at the top of this file, run as
 * the page's kernels in its order (PR #1528, "What it adds": modulated RMSNorm, the bf16
 * projections with fp32 sums, q/k norm and rotary into packed rows, the head-128 attention, the
 * SiLU gate and the gated adds; its precision bullet: bf16 activations and weights, fp32 sums,
 * norms and softmax).  Deterministic: PR #1528, "Measured" (the same step run twice gives
 * identical bytes).  Errors: MI_ERR_INVALID_ARG (layout, pointers), MI_ERR_WORKSPACE (ws too small
 * or misaligned), MI_ERR_CUDA (a launch failed); nothing is enqueued on an argument error.
 *   x        bf16 [B, S, H] input rows (text rows then image tokens)
 *   y        bf16 [B, S, H] output; y == x (in place) is allowed, any other overlap is not
 *   mod      bf16 [B, 6, H]: shift1, scale1, gate1, shift2, scale2, gate2 for batch element b,
 *            applied to every row of that element
 *   rope_cos, rope_sin  fp32 [S, 64] angle tables (element b reads base + b * rope_bstride;
 *            rope_bstride = 0 shares one table); pair p of row s rotates by the angle at [s, p]
 *   key_mask uint8 [B, S]: 0 excludes the key row from attention (padded prompt rows), or NULL.
 *            A query row whose keys are all masked gets a zero attention output.
 *   ws       device workspace of at least mi_block_workspace_size bytes, 256-byte aligned
 *            (cudaMalloc and the PyTorch allocator both give at least that)
 */
mi_status mi_block_forward(mi_block* blk, const mi_seq_layout* L, const void* x, void* y, const void* mod,
                           const float* rope_cos, const float* rope_sin, int rope_bstride,
                           const uint8_t* key_mask, void* ws, size_t ws_bytes, void* stream);

/*
 * mi_block_forward without a caller workspace, for callers that cannot call cudaMalloc: for
 * example a plugin whose host owns every device allocation through its own pool, or code that
 * must not allocate after start-up.  The paper has no counterpart: it is an interface addition.
 *
 * The workspace is a static device array of MI_STATIC_WS_BYTES inside this library, held by every
 * GPU that loads the library until the process exits.  Geometries whose mi_block_workspace_size
 * exceeds it are refused with MI_ERR_WORKSPACE.  Nothing is allocated: no cudaMalloc, cudaFree or
 * allocating library routine.  The first call on a device looks the array's address up
 * (cudaGetSymbolAddress, with that device current); make that first call before any stream
 * capture.  All calls share the one array and it keeps the last call's contents (the block
 * overwrites every intermediate before reading it, so nothing needs clearing); calls that overlap
 * on the GPU (different streams, or different threads without ordering) race on it.  Arguments and
 * results are exactly those of mi_block_forward.
 */
#define MI_STATIC_WS_BYTES ((size_t)64 << 20)
mi_status mi_block_forward_static_ws(mi_block* blk, const mi_seq_layout* L, const void* x, void* y, const void* mod,
                                     const float* rope_cos, const float* rope_sin, int rope_bstride,
                                     const uint8_t* key_mask, void* stream);

/* ------------------------------------------------------------------------- denoising step --- */

typedef struct mi_model_desc {
  int n_blocks;
  const mi_block_desc* blocks; /* n_blocks descriptors (same geometry) */
  int latent_ch;               /* C: latent channels, multiple of 64 */
  const void* w_in;            /* bf16 [H, C]: latent -> hidden embedding */
  const void* w_out;           /* bf16 [C, H]: hidden -> velocity projection */
} mi_model_desc;

typedef struct mi_model mi_model;

mi_status mi_model_init(mi_model** out, const mi_model_desc* desc);
void mi_model_destroy(mi_model* model);
mi_status mi_model_workspace_size(const mi_model* model, const mi_seq_layout* L, size_t* bytes);

/*
 * One planned workspace for several geometries (PR #2281 "What this changes": the host plans one
 * scratch and serves every geometry inside it; "Measured": a picture whose scratch does not fit is
 * refused with an out-of-memory status and the engine keeps serving, returning the same bytes for
 * the next request).  For each of the n layouts, its need is mi_model_workspace_size; a layout is
 * served when its need is at most budget_bytes.
 *   layouts  HOST array of n layouts (n >= 1)
 *   bytes    out: the largest need among the served layouts (0 when none is served)
 *   served   HOST uint8 [n] or NULL, out: 1 for a served layout, 0 for a refused one
 * Returns MI_OK when at least one layout is served, MI_ERR_WORKSPACE (the out-of-memory refusal)
 * when none is, MI_ERR_INVALID_ARG for a bad layout.  One workspace of *bytes then serves every
 * served layout in mi_denoise_step, in any order; a step whose layout needs more than the
 * workspace it is given is refused with MI_ERR_WORKSPACE before anything is enqueued, and the
 * model, its workspace and the stream stay usable.  Host arithmetic only: nothing is enqueued.
 */
mi_status mi_model_plan(const mi_model* model, const mi_seq_layout* layouts, int n, size_t budget_bytes,
                        size_t* bytes, uint8_t* served);

/*
 * One guided denoising step (PR #2281 "What this changes": the pipeline's schedule and
 * classifier-free guidance with an empty negative prompt; PR #1528 "Measured": Euler steps):
 *   u = latent W_in^T;  x_b = [text_rows_b ; u];  x_b <- every block;
 *   vel_b = (RMSNorm(image rows of x_b) (1 + scale_f) + shift_f) W_out^T;
 *   v = vel_1 + guidance (vel_0 - vel_1) when batch == 2 (element 0 the prompt, 1 the negative),
 *   v = vel_0 when batch == 1;  latent <- latent + dt v.
 *   latent    fp32 [N, C] (N = grid_h * grid_w), the Euler state, updated in place in fp32; the
 *             embedding reads it rounded to bf16.  The velocities stay fp32 (unrounded GEMM sums).
 *   text_rows bf16 [B, T, H]
 *   mods      bf16 [n_blocks, B, 6, H] (per block, as in mi_block_forward)
 *   mod_final bf16 [B, 2, H]: shift_f, scale_f
 *   skip_neg  HOST uint8 [n_blocks] or NULL (read on the host while enqueueing): a nonzero entry
 *             makes the negative element (index 1) bypass that block
 */
mi_status mi_denoise_step(mi_model* model, const mi_seq_layout* L, void* latent, const void* text_rows,
                          const void* mods, const void* mod_final, const float* rope_cos, const float* rope_sin,
                          int rope_bstride, const uint8_t* key_mask, float dt, float guidance,
                          const uint8_t* skip_neg, void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------- device builders --- */
/* The per-step inputs the pages compute on the host (PR #1528 "What it adds": "the config, rotary
 * tables and the timestep's modulation are shared"), computed on the device so a whole guided
 * loop can run without the host. */

/* Rotary tables (fp32 [S, 64], S = text_pad + grid_h * grid_w): pair j < 32 of row s turns by
 * (row position) * theta^(-j/32), pair j >= 32 by (column position) * theta^(-(j-32)/32); text row
 * t has position t on both axes, image token (r, c) has (r, c).  Angles in fp64, stored fp32. */
mi_status mi_rope_tables(int text_pad, int grid_h, int grid_w, float theta, float* rope_cos, float* rope_sin,
                         void* stream);

typedef struct mi_tmod_desc {
  int hidden;          /* H, multiple of 256 */
  int n_blocks;
  const void* w_t1;    /* bf16 [H, 256] */
  const void* w_t2;    /* bf16 [H, H] */
  const void* w_mod;   /* bf16 [(6 n_blocks + 2) H, H]: block i's six vectors (shift1, scale1, gate1,
                          shift2, scale2, gate2) at rows [6 i H, 6 (i + 1) H), then shift_f, scale_f */
} mi_tmod_desc;

typedef struct mi_tmod mi_tmod;

mi_status mi_tmod_init(mi_tmod** out, const mi_tmod_desc* desc);
void mi_tmod_destroy(mi_tmod* tm);
mi_status mi_tmod_workspace_size(const mi_tmod* tm, int batch, size_t* bytes);

/* Timestep -> modulation of every block and of the final norm, on the device:
 *   emb = [cos(1000 t f_k), sin(1000 t f_k)], f_k = 10000^(-k/128), k < 128  (256 values)
 *   c = W_t2 silu(W_t1 emb);  all = W_mod silu(c)
 * with a bf16 rounding after every step.  t: device fp32 [batch]; mods: bf16 [n_blocks, batch, 6, H]
 * (the layout mi_denoise_step reads); mod_final: bf16 [batch, 2, H]. */
mi_status mi_timestep_modulation(mi_tmod* tm, const float* t, int batch, void* mods, void* mod_final, void* ws,
                                 size_t ws_bytes, void* stream);

/* t[i] += dt for i < n (device fp32), so a captured step can advance its own timestep. */
mi_status mi_time_advance(float* t, int n, float dt, void* stream);

/* ------------------------------------------------------------------------ single kernels --- */
/* The steps of the block as separate calls (same kernels mi_block_forward launches). */

/* out[r] = x[r] * rsqrt(mean(x[r]^2) + eps) * (1 + mod[b, scale_row]) + mod[b, shift_row],
 * b = r / seq; x, out [batch * seq, hidden]; mod [batch, 6, hidden].  PR #1528, "What it adds"
 * (the modulated RMSNorm kernel; fp32 norm, bf16 out).  out must not overlap x. */
mi_status mi_mod_rmsnorm(const void* x, const void* mod, int shift_row, int scale_row, void* out, int batch,
                         int seq, int hidden, float eps, void* stream);

/* c[m, n] = sum_k a[m, k] w[n, k] (fp32 sums, bf16 out).  a [m, k], w [n, k], c [m, n];
 * k a multiple of 64, n a multiple of 8.  PR #1528, "What it adds" (the projections are bf16 GEMMs
 * with fp32 sums).  Shapes outside these rules are refused with MI_ERR_UNSUPPORTED. */
mi_status mi_gemm_bf16(const void* a, const void* w, void* c, int m, int n, int k, void* stream);

/* out = resid + mod[b, gate_row] * bf16(a w^T), b = row / seq (the W_o / W_d projections fused
 * with the gated residual).  resid, out [m, n] (out may equal resid).  PR #1528, "What it adds"
 * (a bf16 projection with fp32 sums followed by the gated add kernel); same bytes as mi_gemm_bf16
 * then mi_gated_add. */
mi_status mi_gemm_bf16_gated_residual(const void* a, const void* w, const void* resid, const void* mod,
                                      int gate_row, void* out, int m, int n, int k, int seq, void* stream);

/* m_out[:, j] = silu(bf16(a wg^T)[:, j]) * bf16(a wu^T)[:, j] with w = [wg; wu] of 2*inter rows
 * (the gate/up projection fused with the SiLU gate).  inter a multiple of 128.  PR #1528, "What it
 * adds" (a bf16 projection, then the SiLU-gate kernel the page lists as "situ"); same bytes as
 * mi_gemm_bf16 then mi_silu_gate. */
mi_status mi_gemm_bf16_silu_gate(const void* a, const void* w, void* m_out, int m, int inter, int k,
                                 void* stream);

/* PR #1528, "What it adds" (a bf16 projection, then the q/k norm and rotary kernel).
 * The QKV projection with the q/k RMSNorm + rotary fused into its epilogue: a [batch * seq, H]
 * times w_qkv [3H, H]^T; q and k heads go, normalised and rotated, to qp, kp [batch, heads, seq, 128]
 * (identical bytes to mi_gemm_bf16 followed by mi_qk_norm_rope); the v columns go to columns
 * [2H, 3H) of qkv_v [batch * seq, 3H] (its q/k columns are not written).  H = heads * 128, a multiple
 * of 256. */
mi_status mi_gemm_bf16_qkv_rope(const void* a, const void* w_qkv, const void* q_norm_w, const void* k_norm_w,
                                const float* rope_cos, const float* rope_sin, int rope_bstride, void* qp, void* kp,
                                void* qkv_v, int batch, int seq, int n_heads, float eps, void* stream);

/* Per-head RMSNorm (gains q_norm_w / k_norm_w [128]) and rotary of the q and k columns of
 * qkv [batch * seq, 3H], written to qp, kp [batch, heads, seq, 128].  PR #1528, "What it adds"
 * (the kernel for q/k norm and rotary into packed rows).  Rotary pairs are (2p, 2p+1) and use the
 * table angle at (row, p); the tables are read at base + b * rope_bstride. */
mi_status mi_qk_norm_rope(const void* qkv, const void* q_norm_w, const void* k_norm_w, const float* rope_cos,
                          const float* rope_sin, int rope_bstride, void* qp, void* kp, int batch, int seq,
                          int n_heads, float eps, void* stream);

/* o [batch * seq, heads * 128] = softmax(q k^T / sqrt(128)) v per (batch, head); q = qp, k = kp
 * as written by mi_qk_norm_rope, v read from columns [2H, 3H) of qkv; key_mask as above.
 * PR #1528, "What it adds" and "Shared code" (full, non-causal attention at head dim 128; the
 * softmax in fp32).  qp, kp and qkv must be 16-byte aligned (TMA sources). */
mi_status mi_attention(const void* qp, const void* kp, const void* qkv, const uint8_t* key_mask, void* o,
                       int batch, int seq, int n_heads, void* stream);

/* mi_attention on the schedule mi_block_forward uses: one CTA per SM, each taking an equal share of
 * the (query-tile pair, key tile) steps, so no SM idles in a partial last wave.  A pair of query
 * tiles whose keys are split between two CTAs is finished by the second to arrive, which adds the
 * two partial results (unnormalised output, running max and sum) in a fixed order, so results
 * repeat bit for bit.  With no more query-tile pairs than SMs, or more than 8 per SM, the schedule
 * is one CTA per pair, as in mi_attention.  ws: at least mi_attention_workspace_size bytes,
 * 256-byte aligned (0 bytes, and ws may be NULL, when the schedule is one CTA per pair).  Same
 * page as above. */
mi_status mi_attention_workspace_size(int batch, int seq, int n_heads, size_t* bytes);
mi_status mi_attention_ws(const void* qp, const void* kp, const void* qkv, const uint8_t* key_mask, void* o,
                          int batch, int seq, int n_heads, void* ws, size_t ws_bytes, void* stream);

/* out = x + mod[b, gate_row] * y, b = row / seq; x, y, out [batch * seq, hidden].  PR #1528,
 * "What it adds" (the gated add kernel; fp32 arithmetic, one bf16 rounding).  out may equal x. */
mi_status mi_gated_add(const void* x, const void* y, const void* mod, int gate_row, void* out, int batch,
                       int seq, int hidden, void* stream);

/* m[r, j] = silu(gu[r, j]) * gu[r, inter + j]; gu [rows, 2 * inter], m [rows, inter].
 * silu(z) = z / (1 + exp(-z)).  PR #1528, "What it adds" (the kernel listed as "situ", read as the
 * SiLU gate); PR #2281, "Three findings" prints the SiLU minimum (-0.278 near -1.278). */
mi_status mi_silu_gate(const void* gu, void* m, int rows, int inter, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MI_BLOCK_H */
