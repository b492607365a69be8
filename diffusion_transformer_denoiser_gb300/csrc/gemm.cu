// Projection GEMMs of the block: C[M, N] = A[M, K] * W[N, K]^T, bf16 operands, fp32 sums.
//
// The pages' projections are library bf16 GEMMs with fp32 sums (MOSS-Image transformer on CUDA,
// "What it adds").  Here they run on the 5th-generation tensor cores:
//   * warp 0   : TMA producer, 128-byte-swizzled A and W tiles into a 4-stage shared-memory ring;
//   * warp 1   : issues tcgen05.mma (M=128, N=BN, K=16) into TMEM, the warp convergent and one
//                elected lane per instruction;
//   * warps 2-5: epilogue, TMEM -> registers -> bf16 -> global, with the fused element-wise
//                tails (gated residual add, SiLU gate) applied before the single store.
// Persistent grid (one CTA per SM), tiles walked M-fastest so the A panel stays in L2, and two
// TMEM accumulators so the epilogue of tile i overlaps the main loop of tile i+1.  Fixed tile
// order and fixed K order make every launch bit-identical to the previous one.
#include "mi_internal.h"
#include "ptx.cuh"

namespace mi {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int kThreads = 192;

template <int BN>
struct GemmSmem {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int TOTAL = BAR_OFF + 256 + 1024;  // barriers + alignment slack
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs p) {
  using L = GemmSmem<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_m = (p.M + BM - 1) / BM;
  const int num_n = (EPI == EPI_SILU_GATE) ? (p.N / (BN / 2)) : (p.N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int kblocks = p.K / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int mb = tile % num_m;
        const int nb = tile / num_m;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, DEV_TIMEOUT_GEMM + 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], L::STAGE_BYTES);
          tma_load_2d(sA + stage * L::A_BYTES, &tmA, &full[stage], kb * BK, mb * BM);
          if (EPI == EPI_SILU_GATE) {
            // gate rows [nb*BN/2, +BN/2) and the matching up rows [N + nb*BN/2, +BN/2)
            tma_load_2d(sB + stage * L::B_BYTES, &tmB, &full[stage], kb * BK, nb * (BN / 2));
            tma_load_2d(sB + stage * L::B_BYTES + L::B_BYTES / 2, &tmB, &full[stage], kb * BK,
                        p.N + nb * (BN / 2));
          } else {
            tma_load_2d(sB + stage * L::B_BYTES, &tmB, &full[stage], kb * BK, nb * BN);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every load this thread issued has landed before the CTA exits.  Stages before
      // `stage` were last armed in the current lap (parity `phase`), the others in the previous
      // lap (parity `phase ^ 1`, which a never-armed barrier also reports as complete).
      for (int s = 0; s < STAGES; ++s) {
        mbar_wait_drain(&full[s], (s < stage) ? phase : (phase ^ 1u), p.err, DEV_TIMEOUT_GEMM + 2);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs this role convergently; each MMA and commit is issued by one elected lane.
    constexpr uint32_t idesc = idesc_bf16(BM, BN, false, false);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      if (!mbar_wait_warp(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err, DEV_TIMEOUT_GEMM + 3)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_warp(&full[stage], phase, abort_flag, p.err, DEV_TIMEOUT_GEMM + 4)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sdesc_sw128(smem_u32(sA + stage * L::A_BYTES), 16, 1024);
        const uint64_t bd = sdesc_sw128(smem_u32(sB + stage * L::B_BYTES), 16, 1024);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          // K slice k starts 32 bytes further along the swizzled row (descriptor units: 16 bytes)
          tc_mma_ss_warp(d_tmem, ad + 2u * k, bd + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
        }
        tc_commit_warp(&empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      tc_commit_warp(&tfull[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // drain: all MMAs issued by this warp complete before TMEM is released
    tc_commit_warp(drain);
    mbar_wait_drain(drain, 0, p.err, DEV_TIMEOUT_GEMM + 6);
  } else {
    // ------------------------------------------------------------------ epilogue warps
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int mb = tile % num_m;
      const int nb = tile / num_m;
      if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag, p.err, DEV_TIMEOUT_GEMM + 5)) break;
      tc_fence_after();
      const int row = mb * BM + r_in_tile;
      const bool row_ok = row < p.M;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if (EPI == EPI_SILU_GATE) {
        constexpr int HALF = BN / 2;
#pragma unroll 1
        for (int c = 0; c < HALF / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(t_row + c * 32, g);
          tmem_ld32(t_row + HALF + c * 32, u);
          tmem_ld_wait();
          if (row_ok) {
            const int col0 = nb * HALF + c * 32;
            uint4* dst = reinterpret_cast<uint4*>(p.C + (size_t)row * p.ldc + col0);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = v * 8 + e * 2;
                // round the GEMM outputs to bf16 first, as the unfused path stores them
                const float g0 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(g[i])));
                const float g1 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(g[i + 1])));
                const float u0 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(u[i])));
                const float u1 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(u[i + 1])));
                w[e] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
              }
              dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else if (EPI == EPI_QKV_ROPE && nb * BN < 2 * p.hidden) {
        // q or k columns: the tile holds two whole heads of this row.  Per head: round the sums to
        // bf16 (the QKV projection's rounding point), RMSNorm over the 128 values with the gain,
        // rotate the pairs (2p, 2p+1) by the row's angles, and write the packed head row.  The
        // reductions follow the stand-alone q/k kernel's order exactly (sixteen 8-element fma
        // chains combined by the same butterfly), so fused and unfused results are identical.
        const int which = nb * BN >= p.hidden ? 1 : 0;
        const int head0 = (nb * BN - which * p.hidden) / kHeadDim;
        const __nv_bfloat16* gain = which ? p.wk : p.wq;
        __nv_bfloat16* dst_base = which ? p.kp : p.qp;
        const int b = row_ok ? row / p.seq : 0;
        const int s = row_ok ? row % p.seq : 0;
#pragma unroll 1
        for (int hh = 0; hh < BN / kHeadDim; ++hh) {
          uint32_t r[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(t_row + hh * kHeadDim + c * 32, r + c * 32);
          tmem_ld_wait();
          if (row_ok) {
            float part[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float ss = 0.0f;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float f = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[k * 8 + e])));
                r[k * 8 + e] = __float_as_uint(f);
                ss = fmaf(f, f, ss);
              }
              part[k] = ss;
            }
            float v8[8], w4[4];
#pragma unroll
            for (int k = 0; k < 8; ++k) v8[k] = part[k] + part[k + 8];
#pragma unroll
            for (int k = 0; k < 4; ++k) w4[k] = v8[k] + v8[k + 4];
            const float tot = (w4[0] + w4[2]) + (w4[1] + w4[3]);
            const float rstd = rsqrtf(tot * (1.0f / kHeadDim) + p.eps);
            const float* cr = p.rope_cos + (size_t)b * p.rope_bstride + (size_t)s * (kHeadDim / 2);
            const float* sr = p.rope_sin + (size_t)b * p.rope_bstride + (size_t)s * (kHeadDim / 2);
            uint4* dst = reinterpret_cast<uint4*>(
                dst_base + (((size_t)b * p.heads + head0 + hh) * p.seq + s) * kHeadDim);
#pragma unroll
            for (int v = 0; v < 16; ++v) {  // 8 elements = 4 rotary pairs per 16-byte store
              const uint4 gv = __ldg(reinterpret_cast<const uint4*>(gain) + v);
              const uint32_t gs[4] = {gv.x, gv.y, gv.z, gv.w};
              const float4 c4 = __ldg(reinterpret_cast<const float4*>(cr) + v);
              const float4 s4 = __ldg(reinterpret_cast<const float4*>(sr) + v);
              const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
              const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
              uint32_t w[4];
#pragma unroll
              for (int pr = 0; pr < 4; ++pr) {
                const float a = __uint_as_float(r[v * 8 + 2 * pr]) * rstd * bf16_lo(gs[pr]);
                const float bb = __uint_as_float(r[v * 8 + 2 * pr + 1]) * rstd * bf16_hi(gs[pr]);
                w[pr] = pack_bf16x2(fmaf(a, cs[pr], -bb * sn[pr]), fmaf(a, sn[pr], bb * cs[pr]));
              }
              dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else {
        const int b = row_ok ? row / p.seq : 0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(t_row + c * 32, r);
          tmem_ld_wait();
          const int col0 = nb * BN + c * 32;
          if (EPI == EPI_STORE_F32) {
            if (row_ok && col0 < p.N) {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.C) + (size_t)row * p.ldc + col0);
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                if (col0 + v * 4 < p.N)
                  dst[v] = make_float4(__uint_as_float(r[v * 4 + 0]), __uint_as_float(r[v * 4 + 1]),
                                       __uint_as_float(r[v * 4 + 2]), __uint_as_float(r[v * 4 + 3]));
              }
            }
          } else if (row_ok && col0 < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(p.C + (size_t)row * p.ldc + col0);
            if (EPI == EPI_GATED_RESIDUAL) {
              const uint4* xr = reinterpret_cast<const uint4*>(p.resid + (size_t)row * p.ldr + col0);
              const uint4* gr = reinterpret_cast<const uint4*>(p.gate + (size_t)b * p.gate_bstride + col0);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                if (col0 + v * 8 < p.N) {
                  const uint4 xv = xr[v];
                  const uint4 gv = __ldg(gr + v);
                  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
                  const uint32_t gs[4] = {gv.x, gv.y, gv.z, gv.w};
                  uint32_t w[4];
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int i = v * 8 + e * 2;
                    const float a0 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[i])));
                    const float a1 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[i + 1])));
                    w[e] = pack_bf16x2(fmaf(bf16_lo(gs[e]), a0, bf16_lo(xs[e])),
                                       fmaf(bf16_hi(gs[e]), a1, bf16_hi(xs[e])));
                  }
                  dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                }
              }
            } else {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                if (col0 + v * 8 < p.N) {
                  dst[v] = make_uint4(pack_bf16x2(__uint_as_float(r[v * 8 + 0]), __uint_as_float(r[v * 8 + 1])),
                                      pack_bf16x2(__uint_as_float(r[v * 8 + 2]), __uint_as_float(r[v * 8 + 3])),
                                      pack_bf16x2(__uint_as_float(r[v * 8 + 4]), __uint_as_float(r[v * 8 + 5])),
                                      pack_bf16x2(__uint_as_float(r[v * 8 + 6]), __uint_as_float(r[v * 8 + 7])));
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

template <int BN, int EPI>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int num_sms,
                        cudaStream_t s) {
  using L = GemmSmem<BN>;
  auto kern = gemm_bf16_tn_kernel<BN, EPI>;
  static bool attr_done[kMaxDevices] = {};  // per template instance and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int num_m = (a.M + BM - 1) / BM;
  const int num_n = (EPI == EPI_SILU_GATE) ? (a.N / (BN / 2)) : (a.N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int grid = tiles < num_sms ? tiles : num_sms;
  kern<<<grid, kThreads, L::TOTAL, s>>>(ta, tb, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_launch(int epi, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int num_sms,
                        cudaStream_t s) {
  switch (epi) {
    case EPI_STORE:
      return launch_gemm<256, EPI_STORE>(ta, tb, a, num_sms, s);
    case EPI_GATED_RESIDUAL:
      return launch_gemm<256, EPI_GATED_RESIDUAL>(ta, tb, a, num_sms, s);
    case EPI_SILU_GATE:
      return launch_gemm<256, EPI_SILU_GATE>(ta, tb, a, num_sms, s);
    case EPI_STORE_F32:
      return launch_gemm<256, EPI_STORE_F32>(ta, tb, a, num_sms, s);
    case EPI_QKV_ROPE:
      return launch_gemm<256, EPI_QKV_ROPE>(ta, tb, a, num_sms, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace mi
