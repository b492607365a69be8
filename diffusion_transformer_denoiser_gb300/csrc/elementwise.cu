// HBM-bound kernels of the block: modulated RMSNorm, q/k RMSNorm + rotary pack, gated residual
// add, SiLU gate, and the small glue of a guided denoising step (sequence assembly, guidance +
// Euler update).  The MOSS-Image transformer page lists the first four as its hand-written kernels
// ("modulated RMSNorm, q/k norm and rotary into packed rows, situ [SiLU gate], gated add").
//
// All of them move 16-byte vectors (8 bf16) per thread, reduce in fp32 with a fixed shuffle
// order (so results repeat bit for bit), and round once to bf16 at the output.
#include <stdlib.h>

#include "mi_internal.h"
#include "ptx.cuh"

namespace mi {

namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ f32x2_t f2_mul(f32x2_t a, f32x2_t b) {
  f32x2_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// ------------------------------------------------------------------------------------ adaLN norm
// out[i] = x[in_row(i)] * rsqrt(mean(x^2) + eps) * (1 + scale[b]) + shift[b]; one warp per row.
// Row i of the output reads input row (i / out_seq) * in_seq + in_off + i % out_seq, which lets
// the final norm of a denoising step read only the image rows of each batch element.
//
// Each CTA (one per SM) takes a contiguous range of rows; its warps take every kNormWarps-th row
// of it.  A warp keeps `depth` of its rows in flight as bulk asynchronous copies into its own
// shared-memory slots (one mbarrier each), issued before any arithmetic: at the block's 4130 rows
// every row an SM handles is requested at the start, so the reads stream at full depth from the
// first microsecond instead of ramping up behind register-held loads.  A row is read from its slot
// twice (sum of squares, then the outputs, which go straight to global memory) and the slot is then
// refilled with the warp's row `depth` further on.  The launch is programmatic-dependent: the CTAs start (barrier set-up)
// while the previous kernel in the stream finishes and wait for its results before the first copy.
// The arithmetic and its order (per-lane fp32 sums on two packed lanes, then a fixed shuffle
// butterfly) are fixed: results repeat bit for bit.  NV = hidden / 256 (hidden <= 4096).
constexpr int kNormWarps = 16;
constexpr int kNormSlotBytes = 192 * 1024;        // shared memory for row slots per CTA
constexpr int kNormMaxDepth = 4;

template <int NV>
__global__ void __launch_bounds__(kNormWarps * 32, 1)
    mod_rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ shift,
                       const __nv_bfloat16* __restrict__ scale, int mod_bstride, __nv_bfloat16* __restrict__ out,
                       int rows, int out_seq, int in_seq, int in_off, int hidden, float eps, int depth, int* err,
                       int* zero, int zero_n) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  constexpr uint32_t kRowBytes = NV * 512;
  __shared__ uint64_t bars[kNormWarps * kNormMaxDepth];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r0 = (int)((long long)rows * blockIdx.x / gridDim.x);
  const int r1 = (int)((long long)rows * (blockIdx.x + 1) / gridDim.x);
  const int n_mine = (r1 - r0 - warp + kNormWarps - 1) / kNormWarps;  // rows r0 + warp + k * kNormWarps
  uint64_t* my_bars = bars + warp * kNormMaxDepth;
  uint8_t* my_slots = smem_raw + (size_t)warp * depth * kRowBytes;
  if (lane == 0) {
    for (int i = 0; i < depth; ++i) mbar_init(&my_bars[i], 1);
    if (warp == 0) abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  grid_dep_wait();  // x may be the previous kernel's output
  if (zero != nullptr)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < zero_n; i += gridDim.x * blockDim.x) zero[i] = 0;

  auto issue = [&](int k) {  // lane 0: row k of this warp into slot k % depth
    const int r = r0 + warp + k * kNormWarps;
    const int in_row = (r / out_seq) * in_seq + in_off + r % out_seq;
    const int sl = k % depth;
    mbar_arrive_expect_tx(&my_bars[sl], kRowBytes);
    bulk_load(my_slots + (size_t)sl * kRowBytes, x + (size_t)in_row * hidden, kRowBytes, &my_bars[sl]);
  };
  int issued = n_mine < depth ? (n_mine > 0 ? n_mine : 0) : depth;
  if (lane == 0)
    for (int k = 0; k < issued; ++k) issue(k);
  grid_dep_launch();

  // Rows are taken two at a time when a warp has two left (they share one read of the modulation
  // vectors), else one at a time.
  auto row_rstd = [&](const uint4* src) {
    f32x2_t ss2 = 0ull;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const uint4 v = src[i * 32 + lane];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const f32x2_t f = f2_pack(bf16_lo(w[e]), bf16_hi(w[e]));
        ss2 = f2_fma(f, f, ss2);
      }
    }
    float ss_lo, ss_hi;
    f2_unpack(ss2, ss_lo, ss_hi);
    float ss = ss_lo + ss_hi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    return rsqrtf(ss / (float)hidden + eps);
  };
  auto mod_piece = [&](uint4 v, uint4 vs, uint4 vc, f32x2_t rstd2) {
    const f32x2_t one2 = f2_pack(1.0f, 1.0f);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w}, ws[4] = {vs.x, vs.y, vs.z, vs.w}, wc[4] = {vc.x, vc.y, vc.z, vc.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const f32x2_t t = f2_mul(f2_pack(bf16_lo(w[e]), bf16_hi(w[e])), rstd2);
      const f32x2_t c = f2_add(f2_pack(bf16_lo(wc[e]), bf16_hi(wc[e])), one2);
      float lo, hi;
      f2_unpack(f2_fma(t, c, f2_pack(bf16_lo(ws[e]), bf16_hi(ws[e]))), lo, hi);
      o[e] = pack_bf16x2(lo, hi);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  int k = 0;
  while (k < n_mine) {
    const int take = (depth >= 2 && k + 1 < n_mine && (r0 + warp + k * kNormWarps) / out_seq ==
                                            (r0 + warp + (k + 1) * kNormWarps) / out_seq) ? 2 : 1;
    const int slA = k % depth, slB = (k + 1) % depth;
    if (!mbar_wait_warp(&my_bars[slA], (uint32_t)((k / depth) & 1), &abort_flag, err, DEV_TIMEOUT_NORM + 1)) break;
    if (take == 2 &&
        !mbar_wait_warp(&my_bars[slB], (uint32_t)(((k + 1) / depth) & 1), &abort_flag, err, DEV_TIMEOUT_NORM + 1))
      break;
    const uint4* srcA = reinterpret_cast<const uint4*>(my_slots + (size_t)slA * kRowBytes);
    const uint4* srcB = reinterpret_cast<const uint4*>(my_slots + (size_t)slB * kRowBytes);
    const int rowA = r0 + warp + k * kNormWarps;
    const int rowB = rowA + kNormWarps;
    const float rstdA = row_rstd(srcA);
    const float rstdB = take == 2 ? row_rstd(srcB) : 0.0f;
    const int b = rowA / out_seq;
    const uint4* sh = reinterpret_cast<const uint4*>(shift + (size_t)b * mod_bstride);
    const uint4* sc = reinterpret_cast<const uint4*>(scale + (size_t)b * mod_bstride);
    uint4* orowA = reinterpret_cast<uint4*>(out + (size_t)rowA * hidden);
    uint4* orowB = reinterpret_cast<uint4*>(out + (size_t)rowB * hidden);
    const f32x2_t rA = f2_pack(rstdA, rstdA), rB = f2_pack(rstdB, rstdB);
#pragma unroll
    for (int i = 0; i < NV; ++i) {  // each row read again from its slot; (x * rstd) * (1 + scale) + shift
      const uint4 vs = __ldg(sh + i * 32 + lane);
      const uint4 vc = __ldg(sc + i * 32 + lane);
      orowA[i * 32 + lane] = mod_piece(srcA[i * 32 + lane], vs, vc, rA);
      if (take == 2) orowB[i * 32 + lane] = mod_piece(srcB[i * 32 + lane], vs, vc, rB);
    }
    __syncwarp();  // every lane is done with the slots before they are refilled
    for (int t = 0; t < take; ++t) {
      if (k + depth < n_mine) {
        if (lane == 0) {
          fence_proxy_async_smem();
          issue(k + depth);
        }
        ++issued;
      }
      ++k;
    }
  }
  // after an abort: the copies still in flight land before the CTA's shared memory is released
  if (lane == 0)
    for (int j = k; j < issued; ++j)
      mbar_wait_drain(&my_bars[j % depth], (uint32_t)((j / depth) & 1), err, DEV_TIMEOUT_NORM + 2);
}

template <int NV>
cudaError_t mod_rmsnorm_launch_nv(const __nv_bfloat16* x, const __nv_bfloat16* shift, const __nv_bfloat16* scale,
                                  int mod_bstride, __nv_bfloat16* out, int rows, int out_seq, int in_seq, int in_off,
                                  int hidden, float eps, int* err, int num_sms, int dev, cudaStream_t s, int* zero,
                                  int zero_n) {
  constexpr int kRowBytes = NV * 512;
  const int depth_fit = kNormSlotBytes / (kNormWarps * kRowBytes);
  const int depth = depth_fit < kNormMaxDepth ? depth_fit : kNormMaxDepth;
  const int smem = kNormWarps * depth * kRowBytes;
  static bool attr_done[kMaxDevices] = {};
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(mod_rmsnorm_kernel<NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int need = (rows + kNormWarps - 1) / kNormWarps;
  const int grid = need < num_sms ? need : num_sms;
  return launch_kernel(mod_rmsnorm_kernel<NV>, dim3(grid), dim3(kNormWarps * 32), smem, s, true, x, shift, scale,
                       mod_bstride, out, rows, out_seq, in_seq, in_off, hidden, eps, depth, err, zero, zero_n);
}

cudaError_t mod_rmsnorm_any(const __nv_bfloat16* x, const __nv_bfloat16* shift, const __nv_bfloat16* scale,
                            int mod_bstride, __nv_bfloat16* out, int rows, int out_seq, int in_seq, int in_off,
                            int hidden, float eps, int* err, cudaStream_t s, int* zero, int zero_n) {
  static int sms_cache[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (sms_cache[dev] == 0) {
    e = cudaDeviceGetAttribute(&sms_cache[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  if (rows <= 0) return cudaSuccess;
  switch (hidden >> 8) {
#define MI_NORM_CASE(n)                                                                                          \
  case n:                                                                                                        \
    return mod_rmsnorm_launch_nv<n>(x, shift, scale, mod_bstride, out, rows, out_seq, in_seq, in_off, hidden, eps, \
                                    err, sms_cache[dev], dev, s, zero, zero_n);
    MI_NORM_CASE(1) MI_NORM_CASE(2) MI_NORM_CASE(3) MI_NORM_CASE(4) MI_NORM_CASE(5) MI_NORM_CASE(6) MI_NORM_CASE(7)
    MI_NORM_CASE(8) MI_NORM_CASE(9) MI_NORM_CASE(10) MI_NORM_CASE(11) MI_NORM_CASE(12) MI_NORM_CASE(13)
    MI_NORM_CASE(14) MI_NORM_CASE(15) MI_NORM_CASE(16)
#undef MI_NORM_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------------------------------------------ q/k pack
// One warp per (row, head): lanes 0-15 take q, lanes 16-31 take k, 8 consecutive elements each
// (4 rotary pairs).  RMSNorm over the 128 elements of the head, gain, then the rotation of the
// interleaved pairs (2p, 2p+1) by the table angle at (row, p).  Output rows are packed per head:
// qp/kp[(b * heads + h) * S + s][0..128).
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(const __nv_bfloat16* __restrict__ qkv,
                                                           const __nv_bfloat16* __restrict__ wq,
                                                           const __nv_bfloat16* __restrict__ wk,
                                                           const float* __restrict__ cosv,
                                                           const float* __restrict__ sinv, int rope_bstride,
                                                           __nv_bfloat16* __restrict__ qp,
                                                           __nv_bfloat16* __restrict__ kp, int batch, int seq,
                                                           int heads, float eps) {
  const long long item = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long total = (long long)batch * seq * heads;
  if (item >= total) return;
  const int h = (int)(item % heads);
  const long long row = item / heads;  // b * seq + s
  const int b = (int)(row / seq);
  const int s = (int)(row % seq);
  const int H = heads * kHeadDim;
  const int which = lane >> 4;  // 0: q, 1: k
  const int sub = lane & 15;
  const int e0 = sub * 8;
  const uint4 v = *reinterpret_cast<const uint4*>(qkv + (size_t)row * 3 * H + (size_t)which * H +
                                                  (size_t)h * kHeadDim + e0);
  float f[8];
  unpack8(v, f);
  float ss = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float rstd = rsqrtf(ss * (1.0f / kHeadDim) + eps);
  float g[8];
  unpack8(__ldg(reinterpret_cast<const uint4*>((which ? wk : wq) + e0)), g);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = f[e] * rstd * g[e];
  const float* cr = cosv + (size_t)b * rope_bstride + (size_t)s * (kHeadDim / 2) + sub * 4;
  const float* sr = sinv + (size_t)b * rope_bstride + (size_t)s * (kHeadDim / 2) + sub * 4;
  const float4 c4 = __ldg(reinterpret_cast<const float4*>(cr));
  const float4 s4 = __ldg(reinterpret_cast<const float4*>(sr));
  const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
  const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
  float o[8];
#pragma unroll
  for (int pr = 0; pr < 4; ++pr) {
    const float a = f[2 * pr], bb = f[2 * pr + 1];
    o[2 * pr] = fmaf(a, cs[pr], -bb * sn[pr]);
    o[2 * pr + 1] = fmaf(a, sn[pr], bb * cs[pr]);
  }
  __nv_bfloat16* dst = (which ? kp : qp) + (((size_t)b * heads + h) * seq + s) * kHeadDim + e0;
  *reinterpret_cast<uint4*>(dst) = pack8(o);
}

// ------------------------------------------------------------------------------------ gated add
// out = x + gate[b] * y (fp32 fma, one rounding); the same expression as the fused GEMM epilogue.
__global__ void __launch_bounds__(256) gated_add_kernel(const __nv_bfloat16* __restrict__ x,
                                                        const __nv_bfloat16* __restrict__ y,
                                                        const __nv_bfloat16* __restrict__ gate, int gate_bstride,
                                                        __nv_bfloat16* __restrict__ out, long long n_vec, int seq,
                                                        int hidden) {
  const int vpr = hidden >> 3;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / vpr;
    const int cv = (int)(i % vpr);
    const int b = (int)(row / seq);
    float fx[8], fy[8], fg[8];
    unpack8(reinterpret_cast<const uint4*>(x)[i], fx);
    unpack8(reinterpret_cast<const uint4*>(y)[i], fy);
    unpack8(__ldg(reinterpret_cast<const uint4*>(gate + (size_t)b * gate_bstride) + cv), fg);
#pragma unroll
    for (int e = 0; e < 8; ++e) fx[e] = fmaf(fg[e], fy[e], fx[e]);
    reinterpret_cast<uint4*>(out)[i] = pack8(fx);
  }
}

// ------------------------------------------------------------------------------------ SiLU gate
// m[r, j] = silu(gu[r, j]) * gu[r, I + j]; the same expression as the fused GEMM epilogue.
__global__ void __launch_bounds__(256) silu_gate_kernel(const __nv_bfloat16* __restrict__ gu,
                                                        __nv_bfloat16* __restrict__ m, long long n_vec, int inter) {
  const int vpr = inter >> 3;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / vpr;
    const int cv = (int)(i % vpr);
    const uint4* src = reinterpret_cast<const uint4*>(gu + (size_t)row * 2 * inter);
    float g[8], u[8];
    unpack8(src[cv], g);
    unpack8(src[vpr + cv], u);
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = silu_f(g[e]) * u[e];
    reinterpret_cast<uint4*>(m)[i] = pack8(g);
  }
}

// ------------------------------------------------------------------------------------ step glue
// x[b, t] = text[b, t] for t < T, x[b, T + n] = u[n] (the embedded latent is shared by the batch).
__global__ void __launch_bounds__(256) assemble_seq_kernel(const uint4* __restrict__ text, const uint4* __restrict__ u,
                                                           uint4* __restrict__ x, int batch, int text_pad,
                                                           int n_img, int vpr) {
  const long long S = text_pad + n_img;
  const long long total = (long long)batch * S * vpr;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / vpr;
    const int cv = (int)(i % vpr);
    const int b = (int)(row / S);
    const int s = (int)(row % S);
    x[i] = s < text_pad ? text[((long long)b * text_pad + s) * vpr + cv] : u[(long long)(s - text_pad) * vpr + cv];
  }
}

__global__ void __launch_bounds__(256) copy_vec_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                       long long n_vec) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// v = v_neg + g (v_pos - v_neg), latent <- latent + dt v, all fp32.  vel is [batch, N, C].
__global__ void __launch_bounds__(256) cfg_euler_kernel(const float* __restrict__ vel, float* __restrict__ latent,
                                                        long long n, float dt, float guidance, int batch) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float vp = vel[i];
    const float v = batch > 1 ? fmaf(guidance, vp - vel[n + i], vel[n + i]) : vp;
    latent[i] = fmaf(dt, v, latent[i]);
  }
}

__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                                                          long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

// ------------------------------------------------------------------------------------ builders
// Rotary tables on the device: row s, pair j turns by pos * theta^(-(j mod 32)/32) with pos the row
// position (pairs < 32) or column position (pairs >= 32) of the token; text row t has position t
// on both axes.  Angles in fp64, stored as fp32.
__global__ void __launch_bounds__(256) rope_table_kernel(float* __restrict__ cosv, float* __restrict__ sinv, int S,
                                                          int text_pad, int grid_w, double theta) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= S * 64) return;
  const int s = i >> 6;
  const int j = i & 63;
  double pos;
  if (s < text_pad) {
    pos = (double)s;
  } else {
    const int r = (s - text_pad) / grid_w;
    const int c = (s - text_pad) % grid_w;
    pos = (double)(j < 32 ? r : c);
  }
  const double ang = pos * pow(theta, -(double)(j & 31) / 32.0);
  cosv[i] = (float)cos(ang);
  sinv[i] = (float)sin(ang);
}

// Sinusoidal timestep embedding: out[b, k] = cos(scale t_b f_k), out[b, half + k] = sin(scale t_b f_k),
// f_k = max_period^(-k / half); fp64, rounded to bf16.
__global__ void __launch_bounds__(256) timestep_embedding_kernel(const float* __restrict__ t, __nv_bfloat16* __restrict__ out,
                                                                 int batch, int half, double scale, double max_period) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= batch * half) return;
  const int b = i / half;
  const int k = i % half;
  const double ang = scale * (double)t[b] * pow(max_period, -(double)k / (double)half);
  out[(size_t)b * 2 * half + k] = __float2bfloat16_rn((float)cos(ang));
  out[(size_t)b * 2 * half + half + k] = __float2bfloat16_rn((float)sin(ang));
}

__global__ void __launch_bounds__(256) silu_inplace_kernel(__nv_bfloat16* __restrict__ v, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    v[i] = __float2bfloat16_rn(silu_f(__bfloat162float(v[i])));
}

// all[b, (6 i + k) H + c] -> mods[i, b, k, c]; all[b, (6 n + k) H + c] -> final[b, k, c].
__global__ void __launch_bounds__(256) modulation_split_kernel(const uint4* __restrict__ all, uint4* __restrict__ mods,
                                                               uint4* __restrict__ fin, int batch, int n_blocks,
                                                               int vpr /* H / 8 */) {
  const long long per_b = (long long)(6 * n_blocks + 2) * vpr;
  const long long total = per_b * batch;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / per_b);
    const long long r = i % per_b;
    const int vec = (int)(r / vpr);  // which H-wide vector
    const int c = (int)(r % vpr);
    if (vec < 6 * n_blocks) {
      const int blk = vec / 6, k = vec % 6;
      mods[(((long long)blk * batch + b) * 6 + k) * vpr + c] = all[i];
    } else {
      fin[((long long)b * 2 + (vec - 6 * n_blocks)) * vpr + c] = all[i];
    }
  }
}

__global__ void time_advance_kernel(float* __restrict__ t, int n, float dt) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) t[i] += dt;
}

int grid_for(long long work_items, int threads) {
  long long g = (work_items + threads - 1) / threads;
  const long long cap = 152LL * 16;  // enough resident blocks for a grid-stride loop
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("MI_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

cudaError_t mod_rmsnorm_launch(const __nv_bfloat16* x, const __nv_bfloat16* shift, const __nv_bfloat16* scale,
                               int mod_bstride, __nv_bfloat16* out, int rows, int seq, int hidden, float eps, int* err,
                               cudaStream_t s, int* zero, int zero_n) {
  return mod_rmsnorm_any(x, shift, scale, mod_bstride, out, rows, seq, seq, 0, hidden, eps, err, s, zero, zero_n);
}

cudaError_t mod_rmsnorm_rows_launch(const __nv_bfloat16* x, const __nv_bfloat16* shift, const __nv_bfloat16* scale,
                                    int mod_bstride, __nv_bfloat16* out, int rows, int out_seq, int in_seq, int in_off,
                                    int hidden, float eps, int* err, cudaStream_t s) {
  return mod_rmsnorm_any(x, shift, scale, mod_bstride, out, rows, out_seq, in_seq, in_off, hidden, eps, err, s,
                         nullptr, 0);
}

cudaError_t qk_norm_rope_launch(const __nv_bfloat16* qkv, const __nv_bfloat16* wq, const __nv_bfloat16* wk,
                                const float* cos, const float* sin, int rope_bstride, __nv_bfloat16* qp,
                                __nv_bfloat16* kp, int batch, int seq, int n_heads, float eps, cudaStream_t s) {
  const long long warps = (long long)batch * seq * n_heads;
  if (warps <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  qk_norm_rope_kernel<<<(unsigned)blocks, threads, 0, s>>>(qkv, wq, wk, cos, sin, rope_bstride, qp, kp, batch, seq,
                                                           n_heads, eps);
  return cudaGetLastError();
}

cudaError_t gated_add_launch(const __nv_bfloat16* x, const __nv_bfloat16* y, const __nv_bfloat16* gate,
                             int gate_bstride, __nv_bfloat16* out, int rows, int seq, int hidden, cudaStream_t s) {
  const long long n_vec = (long long)rows * hidden / 8;
  if (n_vec <= 0) return cudaSuccess;
  gated_add_kernel<<<grid_for(n_vec, 256), 256, 0, s>>>(x, y, gate, gate_bstride, out, n_vec, seq, hidden);
  return cudaGetLastError();
}

cudaError_t silu_gate_launch(const __nv_bfloat16* gu, __nv_bfloat16* m, int rows, int inter, cudaStream_t s) {
  const long long n_vec = (long long)rows * inter / 8;
  if (n_vec <= 0) return cudaSuccess;
  silu_gate_kernel<<<grid_for(n_vec, 256), 256, 0, s>>>(gu, m, n_vec, inter);
  return cudaGetLastError();
}

cudaError_t assemble_seq_launch(const __nv_bfloat16* text, const __nv_bfloat16* u, __nv_bfloat16* x, int batch,
                                int text_pad, int n_img, int hidden, cudaStream_t s) {
  const int vpr = hidden / 8;
  const long long total = (long long)batch * (text_pad + n_img) * vpr;
  if (total <= 0) return cudaSuccess;
  assemble_seq_kernel<<<grid_for(total, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(text),
                                                            reinterpret_cast<const uint4*>(u),
                                                            reinterpret_cast<uint4*>(x), batch, text_pad, n_img, vpr);
  return cudaGetLastError();
}

cudaError_t copy_rows_launch(const __nv_bfloat16* src, __nv_bfloat16* dst, size_t n_elems, cudaStream_t s) {
  const long long n_vec = (long long)(n_elems / 8);
  if (n_vec <= 0) return cudaSuccess;
  copy_vec_kernel<<<grid_for(n_vec, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(src),
                                                        reinterpret_cast<uint4*>(dst), n_vec);
  return cudaGetLastError();
}

cudaError_t cfg_euler_launch(const float* vel, float* latent, int n_img, int channels, float dt, float guidance,
                             int batch, cudaStream_t s) {
  const long long n = (long long)n_img * channels;
  if (n <= 0) return cudaSuccess;
  cfg_euler_kernel<<<grid_for(n, 256), 256, 0, s>>>(vel, latent, n, dt, guidance, batch);
  return cudaGetLastError();
}

cudaError_t rope_table_launch(float* cosv, float* sinv, int S, int text_pad, int grid_w, double theta, cudaStream_t s) {
  if (S <= 0) return cudaSuccess;
  rope_table_kernel<<<(S * 64 + 255) / 256, 256, 0, s>>>(cosv, sinv, S, text_pad, grid_w, theta);
  return cudaGetLastError();
}

cudaError_t timestep_embedding_launch(const float* t, __nv_bfloat16* out, int batch, int dim, double scale,
                                      double max_period, cudaStream_t s) {
  const int half = dim / 2;
  timestep_embedding_kernel<<<(batch * half + 255) / 256, 256, 0, s>>>(t, out, batch, half, scale, max_period);
  return cudaGetLastError();
}

cudaError_t silu_inplace_launch(__nv_bfloat16* v, long long n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  silu_inplace_kernel<<<grid_for(n, 256), 256, 0, s>>>(v, n);
  return cudaGetLastError();
}

cudaError_t modulation_split_launch(const __nv_bfloat16* all, __nv_bfloat16* mods, __nv_bfloat16* fin, int batch,
                                    int n_blocks, int hidden, cudaStream_t s) {
  const long long total = (long long)batch * (6 * n_blocks + 2) * (hidden / 8);
  modulation_split_kernel<<<grid_for(total, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(all),
                                                               reinterpret_cast<uint4*>(mods),
                                                               reinterpret_cast<uint4*>(fin), batch, n_blocks,
                                                               hidden / 8);
  return cudaGetLastError();
}

cudaError_t time_advance_launch(float* t, int n, float dt, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  time_advance_kernel<<<(n + 255) / 256, 256, 0, s>>>(t, n, dt);
  return cudaGetLastError();
}

cudaError_t f32_to_bf16_launch(const float* src, __nv_bfloat16* dst, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  f32_to_bf16_kernel<<<grid_for((long long)n, 256), 256, 0, s>>>(src, dst, (long long)n);
  return cudaGetLastError();
}

}  // namespace mi
