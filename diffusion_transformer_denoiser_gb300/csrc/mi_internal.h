// Internal declarations shared by the launch layer and the kernels (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mi {

constexpr int kMaxDevices = 64;
constexpr int kHeadDim = 128;

enum GemmEpilogue : int {
  EPI_STORE = 0,           // C = A W^T
  EPI_GATED_RESIDUAL = 1,  // C = resid + gate[b] * bf16(A W^T)
  EPI_SILU_GATE = 2,       // C[:, j] = silu(bf16(A Wg^T)[:, j]) * bf16(A Wu^T)[:, j], W = [Wg; Wu]
  EPI_STORE_F32 = 3,       // C (fp32) = A W^T, the fp32 sums unrounded (C is a float*, ldc in floats)
  EPI_QKV_ROPE = 4,        // QKV projection: q/k columns -> per-head RMSNorm + rotary -> qp/kp packed
                           // [B, heads, S, 128]; v columns -> C (the q/k columns of C are not written)
};

struct GemmArgs {
  int M, N, K;              // for EPI_SILU_GATE, N is the width of the output (I), W has 2N rows
  __nv_bfloat16* C;
  int ldc;
  const __nv_bfloat16* resid;  // EPI_GATED_RESIDUAL: [M, ldr]
  int ldr;
  const __nv_bfloat16* gate;   // EPI_GATED_RESIDUAL: gate of batch b at gate + b * gate_bstride
  int gate_bstride;
  int seq;                     // rows per batch element (selects the gate vector / rotary row)
  int* err;                    // device error flag
  // EPI_QKV_ROPE
  __nv_bfloat16* qp;
  __nv_bfloat16* kp;
  const __nv_bfloat16* wq;     // [128] q RMSNorm gain
  const __nv_bfloat16* wk;     // [128] k RMSNorm gain
  const float* rope_cos;       // [S, 64] per batch element at b * rope_bstride
  const float* rope_sin;
  int rope_bstride;
  int hidden;                  // H (q columns [0, H), k columns [H, 2H))
  int heads;
  float eps;
  // Stream-K tail (EPI_STORE, EPI_GATED_RESIDUAL, EPI_STORE_F32): scratch of gemm_sk_scratch_bytes()
  // bytes (256-byte aligned) or null, which keeps the plain persistent schedule.  The launcher fills
  // in the three fields below.
  void* sk_scratch;
  int* sk_count;               // [8 * SMs] arrival counters (one per 32-row quarter of a tail tile)
  float* sk_partial;           // [2 * SMs][256 columns][128 rows] fp32 partial tiles, two slots per CTA
  int sk_tiles;                // tiles on the stream-K tail (0: none)
  int half_from;               // CTA-pair kernel: tiles from this index on run as two half-width tiles
                               // each (set by the launcher)
};

cudaError_t gemm_launch(int epi, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int num_sms,
                        cudaStream_t s);
// Scratch bytes the stream-K tail of this GEMM needs (0 when the plain schedule is used for it).
size_t gemm_sk_scratch_bytes(int epi, int M, int N, int K, int num_sms);

struct AttnArgs {
  int batch, seq, n_heads;
  const uint8_t* key_mask;     // [B, S] or null
  __nv_bfloat16* out;          // [B, S, n_heads * 128]
  float scale_log2;            // log2(e) / sqrt(128)
  int* err;
  // Scratch of attention_scratch_bytes() (256-byte aligned) or null.  With it the grid is one CTA
  // per SM and units may be split between neighbouring CTAs; without it, one CTA per unit.
  float* part;                 // partial results of split units, two slots per CTA
  int* count;                  // [units][2] arrival counters, zero at launch (left zero after it)
};

// q/k maps: 3-D over (128, S, B * n_heads); v map: 4-D over (128, n_heads, S, B) of the qkv buffer.
cudaError_t attention_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const AttnArgs& a, int num_sms, cudaStream_t s);
// CTAs of a launch (num_sms <= 0: one per unit, no splits).
int attention_grid(int batch, int seq, int n_heads, int num_sms);
// Scratch bytes of the split schedule (0 when there are no more units than SMs), and the bytes of
// its arrival counters, which come first.
size_t attention_scratch_bytes(int batch, int seq, int n_heads, int num_sms);
size_t attention_count_bytes(int batch, int seq, int n_heads);

// Element-wise kernels (elementwise.cu).
// zero/zero_n: an int array the kernel clears (after the previous kernel in the stream is done),
// for counters a later kernel of the same forward needs at zero; null for none.
cudaError_t mod_rmsnorm_launch(const __nv_bfloat16* x, const __nv_bfloat16* shift, const __nv_bfloat16* scale,
                               int mod_bstride, __nv_bfloat16* out, int rows, int seq, int hidden, float eps,
                               int* err, cudaStream_t s, int* zero = nullptr, int zero_n = 0);
cudaError_t qk_norm_rope_launch(const __nv_bfloat16* qkv, const __nv_bfloat16* wq, const __nv_bfloat16* wk,
                                const float* cos, const float* sin, int rope_bstride, __nv_bfloat16* qp,
                                __nv_bfloat16* kp, int batch, int seq, int n_heads, float eps, cudaStream_t s);
cudaError_t gated_add_launch(const __nv_bfloat16* x, const __nv_bfloat16* y, const __nv_bfloat16* gate,
                             int gate_bstride, __nv_bfloat16* out, int rows, int seq, int hidden, cudaStream_t s);
cudaError_t silu_gate_launch(const __nv_bfloat16* gu, __nv_bfloat16* m, int rows, int inter, cudaStream_t s);
cudaError_t assemble_seq_launch(const __nv_bfloat16* text, const __nv_bfloat16* u, __nv_bfloat16* x, int batch,
                                int text_pad, int n_img, int hidden, cudaStream_t s);
cudaError_t mod_rmsnorm_rows_launch(const __nv_bfloat16* x, const __nv_bfloat16* shift, const __nv_bfloat16* scale,
                                    int mod_bstride, __nv_bfloat16* out, int rows, int out_seq, int in_seq, int in_off,
                                    int hidden, float eps, int* err, cudaStream_t s);
cudaError_t copy_rows_launch(const __nv_bfloat16* src, __nv_bfloat16* dst, size_t n_elems, cudaStream_t s);
cudaError_t cfg_euler_launch(const float* vel, float* latent, int n_img, int channels, float dt, float guidance,
                             int batch, cudaStream_t s);
cudaError_t f32_to_bf16_launch(const float* src, __nv_bfloat16* dst, size_t n, cudaStream_t s);
cudaError_t rope_table_launch(float* cosv, float* sinv, int S, int text_pad, int grid_w, double theta, cudaStream_t s);
cudaError_t timestep_embedding_launch(const float* t, __nv_bfloat16* out, int batch, int dim, double scale,
                                      double max_period, cudaStream_t s);
cudaError_t silu_inplace_launch(__nv_bfloat16* v, long long n, cudaStream_t s);
cudaError_t modulation_split_launch(const __nv_bfloat16* all, __nv_bfloat16* mods, __nv_bfloat16* fin, int batch,
                                    int n_blocks, int hidden, cudaStream_t s);
cudaError_t time_advance_launch(float* t, int n, float dt, cudaStream_t s);

// Programmatic dependent launch (PDL): a kernel launched with it may start its prologue while the
// previous kernel in the stream is still running; it waits in griddepcontrol.wait before its first
// global-memory access.  On unless the environment sets MI_PDL=0 (read once per process).
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (pdl && pdl_enabled()) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Self-test of the bounded pipeline waits (selftest.cu).
cudaError_t wait_timeout_selftest_launch(int* err, unsigned long long limit_ns, cudaStream_t s);

// Tensor maps (api.cu).
bool encode_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                    uint32_t box_inner, uint32_t box_rows);
bool encode_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                    uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);
bool encode_4d_bf16(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                    const uint32_t box[4]);

}  // namespace mi
