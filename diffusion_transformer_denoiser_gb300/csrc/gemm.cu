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
//
// Stream-K tail: when the tile count is not a multiple of the grid, the last partial wave would
// leave SMs idle.  Instead, the last full wave and the remainder ("tail tiles", or all tiles when
// there are fewer tiles than SMs) have their k-blocks spread evenly over the CTAs, each CTA taking
// its share first.  A share is at least half a tile's k-loop, so a tail tile is split between at
// most three CTAs.  A CTA holding part of a tail tile writes its fp32 partial sums to scratch and
// counts its k-blocks into the tile's arrival counter; the CTA whose count completes the tile adds
// the other parts to its own (still in TMEM) in CTA order, a fixed order, so results still repeat
// bit for bit, and runs the epilogue.  Nobody waits for another CTA: no co-residency is assumed.
#include <stdlib.h>

#include <climits>

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

// Epilogues that support the stream-K tail (their output is a function of each fp32 sum alone).
template <int EPI>
constexpr bool kStreamK = EPI == EPI_STORE || EPI == EPI_GATED_RESIDUAL || EPI == EPI_STORE_F32;

// One unit of work of a CTA: k-blocks [kb0, kb1) of a tile.  slot >= 0 marks a part of a tail
// tile (its partial-sum slot in scratch); tail is the tile's index among the tail tiles.
struct Work {
  int tile, kb0, kb1, slot, tail;
};

// The schedule shared by the producer, MMA and epilogue warps.  Items 0-2 are the tail tiles this
// CTA's share of tail k-blocks touches (a share spans less than two tiles' k-loops, so at most
// three tiles; any may be empty, and a tile the share covers whole is an ordinary item); items from
// 3 on are its whole tiles, strided by the grid.  get() returns 1 for a valid item, 0 for an empty
// one and -1 past the end.
struct Schedule {
  int kblocks, dp_tiles;     // tiles [0, dp_tiles) whole; [dp_tiles, dp_tiles + tail tiles) stream-K
  long long u_begin, u_end;  // this CTA's share of the tail's k-block units

  __device__ Schedule(int num_tiles, int kblocks_, int sk_tiles) : kblocks(kblocks_), dp_tiles(num_tiles - sk_tiles) {
    const long long U = (long long)sk_tiles * kblocks_;
    u_begin = U * blockIdx.x / gridDim.x;
    u_end = U * (blockIdx.x + 1) / gridDim.x;
  }

  __device__ int get(int idx, Work& w) const {
    if (idx < 3) {
      const long long t0 = u_begin / kblocks;
      const long long t = t0 + idx;
      const long long lo = u_begin > t * kblocks ? u_begin : t * kblocks;
      const long long hi = u_end < (t + 1) * kblocks ? u_end : (t + 1) * kblocks;
      if (lo >= hi) return 0;
      w.tile = dp_tiles + (int)t;
      w.kb0 = (int)(lo - t * kblocks);
      w.kb1 = (int)(hi - t * kblocks);
      w.slot = (w.kb0 == 0 && w.kb1 == kblocks) ? -1 : 2 * (int)blockIdx.x + (t == t0 ? 0 : 1);
      w.tail = (int)t;
      return 1;
    }
    const int tile = (int)blockIdx.x + (idx - 3) * (int)gridDim.x;
    if (tile >= dp_tiles) return -1;
    w.tile = tile;
    w.kb0 = 0;
    w.kb1 = kblocks;
    w.slot = -1;
    w.tail = -1;
    return 1;
  }
};

// The CTA whose share of tail units holds unit x (the inverse of u_begin = U * b / grid).
__device__ __forceinline__ int sk_owner(long long x, long long U, int grid) {
  return (int)(((x + 1) * grid - 1) / U);
}

// Inputs of the epilogue of 32 consecutive columns of one row: the residual and gate vectors of
// the gated residual add (nothing for the other stream-K capable epilogues).  All are loaded
// before any store of the chunk: stores to C could alias the residual, so loads placed after them
// would each wait for a round trip of their own.
struct ChunkIn {
  uint4 x[4], g[4];
};

template <int EPI>
__device__ __forceinline__ void load_chunk_in(const GemmArgs& p, int row, int b, int col0, ChunkIn& in) {
  if (EPI == EPI_GATED_RESIDUAL && col0 < p.N) {
    const uint4* xr = reinterpret_cast<const uint4*>(p.resid + (size_t)row * p.ldr + col0);
    const uint4* gr = reinterpret_cast<const uint4*>(p.gate + (size_t)b * p.gate_bstride + col0);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      if (col0 + v * 8 < p.N) {
        in.x[v] = xr[v];
        in.g[v] = __ldg(gr + v);
      }
    }
  }
}

// Epilogue of 32 consecutive fp32 sums (bit patterns in r) of one row for the stream-K capable
// epilogues: plain store, fp32 store, or x + gate[b] * bf16(sum) with x and gate from `in`.
template <int EPI>
__device__ __forceinline__ void store_chunk(const GemmArgs& p, const uint32_t (&r)[32], int row, int col0,
                                            const ChunkIn& in) {
  if (EPI == EPI_STORE_F32) {
    if (col0 < p.N) {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.C) + (size_t)row * p.ldc + col0);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        if (col0 + v * 4 < p.N)
          dst[v] = make_float4(__uint_as_float(r[v * 4 + 0]), __uint_as_float(r[v * 4 + 1]),
                               __uint_as_float(r[v * 4 + 2]), __uint_as_float(r[v * 4 + 3]));
      }
    }
  } else if (col0 < p.N) {
    uint4* dst = reinterpret_cast<uint4*>(p.C + (size_t)row * p.ldc + col0);
    if (EPI == EPI_GATED_RESIDUAL) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (col0 + v * 8 < p.N) {
          const uint32_t xs[4] = {in.x[v].x, in.x[v].y, in.x[v].z, in.x[v].w};
          const uint32_t gs[4] = {in.g[v].x, in.g[v].y, in.g[v].z, in.g[v].w};
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = v * 8 + e * 2;
            const float a0 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[i])));
            const float a1 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[i + 1])));
            w[e] = pack_bf16x2(fmaf(bf16_lo(gs[e]), a0, bf16_lo(xs[e])), fmaf(bf16_hi(gs[e]), a1, bf16_hi(xs[e])));
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

// Epilogue of one tile for the row of TMEM lane (t_row's lane base + lane): the fused element-wise
// tail of each epilogue applied to the fp32 sums, then the single store.  Shared by the one-CTA and
// the CTA-pair kernels (row: this thread's output row; nb: the tile's column block).
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& p, uint32_t t_row, int row, bool row_ok, int nb) {
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
      ChunkIn in;  // loaded before the TMEM read: one wait for memory per chunk
      if (row_ok) load_chunk_in<EPI>(p, row, b, nb * BN + c * 32, in);
      uint32_t r[32];
      tmem_ld32(t_row + c * 32, r);
      tmem_ld_wait();
      if (row_ok) store_chunk<EPI>(p, r, row, nb * BN + c * 32, in);
    }
  }
}

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
  grid_dep_wait();  // the operands may be the previous kernel's outputs
  grid_dep_launch();

  const int num_m = (p.M + BM - 1) / BM;
  const int num_n = (EPI == EPI_SILU_GATE) ? (p.N / (BN / 2)) : (p.N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int kblocks = p.K / BK;
  const Schedule sched(num_tiles, kblocks, kStreamK<EPI> ? p.sk_tiles : 0);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Work w;
      for (int idx = 0, r; ok && (r = sched.get(idx, w)) >= 0; ++idx) {
        if (r == 0) continue;
        const int mb = w.tile % num_m;
        const int nb = w.tile / num_m;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
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
            // the 256-row W tile as two 128-row boxes (W maps have 128-row boxes)
            tma_load_2d(sB + stage * L::B_BYTES, &tmB, &full[stage], kb * BK, nb * BN);
            tma_load_2d(sB + stage * L::B_BYTES + L::B_BYTES / 2, &tmB, &full[stage], kb * BK, nb * BN + BN / 2);
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
    Work w;
    for (int idx = 0, r; ok && (r = sched.get(idx, w)) >= 0; ++idx) {
      if (r == 0) continue;
      if (!mbar_wait_warp(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err, DEV_TIMEOUT_GEMM + 3)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
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
          tc_mma_ss_warp(d_tmem, ad + 2u * k, bd + 2u * k, idesc, (kb > w.kb0 || k != 0) ? 1u : 0u);
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
    Work w;
    for (int idx = 0, rr; (rr = sched.get(idx, w)) >= 0; ++idx) {
      if (rr == 0) continue;
      const int mb = w.tile % num_m;
      const int nb = w.tile / num_m;
      const int row = mb * BM + r_in_tile;
      const bool row_ok = row < p.M;
      if (EPI == EPI_GATED_RESIDUAL && row_ok) {
        // the residual row segment of this tile into L2 while the main loop still runs, so the
        // epilogue's reads do not each wait for HBM
        const __nv_bfloat16* xr = p.resid + (size_t)row * p.ldr + nb * BN;
#pragma unroll
        for (int k = 0; k < BN / 64; ++k)
          if (nb * BN + k * 64 < p.N) asm volatile("prefetch.global.L2 [%0];" ::"l"(xr + k * 64));
      }
      if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag, p.err, DEV_TIMEOUT_GEMM + 5)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if (kStreamK<EPI> && w.slot >= 0) {
        // ---- part of a tail tile: fp32 partial sums of this warp's 32 rows to its scratch slot,
        // laid out as [64 groups of 4 columns][128 rows][4], so that the 32 lanes (consecutive
        // rows) of each 16-byte store write 512 contiguous bytes
        float4* part = reinterpret_cast<float4*>(p.sk_partial + (size_t)w.slot * BM * BN) + r_in_tile;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(t_row + c * 32, v);
          tmem_ld_wait();
          if (row_ok) {
            float4* dst = part + (size_t)c * 8 * BM;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              __stcg(dst + i * BM, make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                               __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
          }
        }
        // count this warp's k-blocks into the arrival counter of its quarter of the tile, the
        // writes above made visible device-wide first
        __threadfence();
        __syncwarp();
        int* cnt = p.sk_count + 4 * w.tail + q;
        int prev = 0;
        if (lane == 0) prev = atomicAdd(cnt, w.kb1 - w.kb0);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev + (w.kb1 - w.kb0) == kblocks) {
          // the last part to arrive: add the other parts (from scratch) and this one (from TMEM)
          // in CTA order, then run the epilogue
          __threadfence();
          const long long U = (long long)p.sk_tiles * kblocks;
          const int b_first = sk_owner((long long)w.tail * kblocks, U, gridDim.x);
          const int b_last = sk_owner((long long)(w.tail + 1) * kblocks - 1, U, gridDim.x);
          const int me = (int)blockIdx.x;
          if (b_last - b_first > 2 && lane == 0) atomicCAS(p.err, 0, DEV_SCHEDULE_GEMM);  // not a host plan
          const float4* src[2] = {nullptr, nullptr};
          int n_other = 0;
          for (int pb = b_first; pb <= b_last && pb <= b_first + 2; ++pb) {
            if (pb == me) continue;
            const int first_tail = (int)((U * pb / gridDim.x) / kblocks);
            const int slot = 2 * pb + (w.tail == first_tail ? 0 : 1);
            src[n_other++] = reinterpret_cast<const float4*>(p.sk_partial + (size_t)slot * BM * BN) + r_in_tile;
          }
          const int my_pos = me - b_first;  // where this CTA's part falls in the order
          const int bb = row_ok ? row / p.seq : 0;
          // n_other and my_pos are the same for the whole warp, so every lane takes the same path
          // to the TMEM reads; row_ok only guards memory accesses.  Columns 4i..4i+3 of a chunk
          // are i * BM float4 past the chunk's first group.  Each chunk issues all its loads (the
          // other parts, the residual and the gate) before the TMEM read, so it waits for memory
          // once.
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float4 x0[8], x1[8];
            ChunkIn in;
            if (row_ok) {
              const float4* s0 = src[0] + (size_t)c * 8 * BM;
#pragma unroll
              for (int i = 0; i < 8; ++i) x0[i] = __ldcg(s0 + i * BM);
              if (n_other > 1) {
                const float4* s1 = src[1] + (size_t)c * 8 * BM;
#pragma unroll
                for (int i = 0; i < 8; ++i) x1[i] = __ldcg(s1 + i * BM);
              }
              load_chunk_in<EPI>(p, row, bb, nb * BN + c * 32, in);
            }
            uint32_t v[32];
            tmem_ld32(t_row + c * 32, v);
            tmem_ld_wait();
            if (row_ok) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float a0[4] = {x0[i].x, x0[i].y, x0[i].z, x0[i].w};
                const float a1[4] = {x1[i].x, x1[i].y, x1[i].z, x1[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  // two parts add the same in either order; three add as (first + second) + third
                  const float own = __uint_as_float(v[4 * i + e]);
                  float t;
                  if (n_other == 1) t = own + a0[e];
                  else if (my_pos == 0) t = (own + a0[e]) + a1[e];
                  else if (my_pos == 1) t = (a0[e] + own) + a1[e];
                  else t = (a0[e] + a1[e]) + own;
                  v[4 * i + e] = __float_as_uint(t);
                }
              }
              store_chunk<EPI>(p, v, row, nb * BN + c * 32, in);
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
        continue;
      }
      epilogue_tile<BN, EPI>(p, t_row, row, row_ok, nb);
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

// ---------------------------------------------------------------------------------------------
// CTA-pair kernel: a cluster of two CTAs computes 256 x 256 tiles with tcgen05 cta_group::2 MMAs.
// Each CTA loads its own 128 rows of A and half of the 256-row W tile (64-column k-blocks), so a
// pipeline stage holds 32 KB per CTA instead of 48 KB: six stages fit where the one-CTA kernel has
// four, and each SM pulls a third less operand data per MMA.  The leader CTA (rank 0) issues the
// MMAs for the pair; each CTA's epilogue drains its own 128 TMEM rows.  A partial last wave of at
// most half the clusters runs as half-width tiles (256 x 128, M=256 N=128 MMAs) on twice as many
// clusters: each CTA still loads a 128-row W box, starting at its 64 rows, and the MMA reads the
// first 64; an element's k-loop is the same in either width, so results do not change.
//   * warp 0 of each CTA: TMA producer into its own ring.  Both CTAs' copies of a stage complete on
//     the leader's `full` barrier (the pair form of the TMA), which the leader arms for both;
//   * warp 1 of the leader: waits on `full`, issues the pair MMAs and commits to `empty` / `tfull`
//     in both CTAs (multicast);
//   * warps 2-5 of each CTA: epilogue, then an arrive on the leader's `tempty` (count 8).
// All waits are bounded.  The leader's producer arms every stage whose release both CTAs see (its
// wait ignores the abort flag), so its drain covers the follower's copies too; both CTAs meet at a
// cluster barrier before TMEM is released and either exits.
constexpr int kPairStages = 6;

struct PairSmem {
  static constexpr int A_BYTES = BM * BK * 2;   // 128 rows of A
  static constexpr int B_BYTES = 128 * BK * 2;  // this CTA's half of the 256-row W tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_OFF = kPairStages * STAGE_BYTES;
  static constexpr int TOTAL = BAR_OFF + 512 + 1024;  // barriers + alignment slack
};

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs p) {
  constexpr int BN = 256;
  using L = PairSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kPairStages * L::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);  // the leader's: both CTAs' copies
  uint64_t* empty = full + kPairStages;
  uint64_t* tfull = empty + kPairStages;     // [2]
  uint64_t* tempty = tfull + 2;              // [2], leader: 4 local + 4 remote epilogue warps
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
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
    tmem_alloc_pair(tmem_slot, 2 * BN);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive or multicast commit
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_wait();  // the operands may be the previous kernel's outputs
  grid_dep_launch();

  const int num_pm = (p.M + 2 * BM - 1) / (2 * BM);
  const int num_n = (EPI == EPI_SILU_GATE) ? (p.N / (BN / 2)) : (p.N + BN - 1) / BN;
  const int num_tiles = num_pm * num_n;
  // Tiles from p.half_from on (the partial last wave) run as two half-width tiles each (N = 128),
  // so the last wave takes half a tile's time on twice as many clusters.
  const int num_units = p.half_from < num_tiles ? num_tiles + (num_tiles - p.half_from) : num_tiles;
  const int kblocks = p.K / BK;
  const int cid = (int)blockIdx.x >> 1;
  const int n_clusters = (int)gridDim.x >> 1;
  // unit u -> tile (pm, nb) and, for a half-width unit, which half (hh = 0, 1; -1 for a whole tile)
  auto decode = [&](int u, int& pm, int& nb, int& hh) {
    int t = u;
    hh = -1;
    if (u >= p.half_from) {
      t = p.half_from + (u - p.half_from) / 2;
      hh = (u - p.half_from) & 1;
    }
    pm = t % num_pm;
    nb = t / num_pm;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer (both CTAs)
      const uint32_t leader_full = cluster_addr(full, 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cid; u < num_units && ok; u += n_clusters) {
        int pm, nb, hh;
        decode(u, pm, nb, hh);
        const int m0 = pm * 2 * BM + (int)rank * BM;
        // W rows of this CTA's half of the unit's columns: 128 for a whole tile, 64 for a half tile
        // (the 128-row box then brings 64 more, which the MMA does not read)
        int b0;
        if (EPI == EPI_SILU_GATE) {
          // the leader loads gate rows, the follower the matching up rows
          b0 = (int)rank * p.N + nb * (BN / 2) + (hh < 0 ? 0 : hh * 64);
        } else {
          b0 = hh < 0 ? nb * BN + (int)rank * 128 : nb * BN + hh * 128 + (int)rank * 64;
        }
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_noabort<true>(&empty[stage], phase ^ 1u, abort_flag, p.err, DEV_TIMEOUT_GEMM + 11)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * L::STAGE_BYTES);
          const uint32_t fb = leader_full + stage * 8;
          tma_load_2d_pair(sA + stage * L::A_BYTES, &tmA, fb, kb * BK, m0);
          tma_load_2d_pair(sB + stage * L::B_BYTES, &tmB, fb, kb * BK, b0);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain (leader): every armed phase, which counts both CTAs' copies, has completed
      if (leader) {
        for (int s = 0; s < kPairStages; ++s) {
          mbar_wait_drain(&full[s], (s < stage) ? phase : (phase ^ 1u), p.err, DEV_TIMEOUT_GEMM + 12);
        }
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ------------------------------------------------------------------ MMA issuer (leader)
      constexpr uint32_t idesc_full = idesc_bf16(2 * BM, BN, false, false);
      constexpr uint32_t idesc_half = idesc_bf16(2 * BM, BN / 2, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = cid; u < num_units && ok; u += n_clusters) {
        if (!mbar_wait_warp<true>(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err, DEV_TIMEOUT_GEMM + 13)) break;
        tc_fence_after();
        const uint32_t idesc = u < p.half_from ? idesc_full : idesc_half;
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_warp<true>(&full[stage], phase, abort_flag, p.err, DEV_TIMEOUT_GEMM + 14)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(sA + stage * L::A_BYTES), 16, 1024);
          const uint64_t bd = sdesc_sw128(smem_u32(sB + stage * L::B_BYTES), 16, 1024);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_pair_warp(d_tmem, ad + 2u * k, bd + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
          tc_commit_pair_warp(&empty[stage]);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        tc_commit_pair_warp(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      tc_commit_pair_warp(drain);
      mbar_wait_drain<true>(drain, 0, p.err, DEV_TIMEOUT_GEMM + 16);
    } else if (lane == 0) {
      // follower: the leader's last commit (multicast to this CTA too) lands before this CTA exits
      mbar_wait_drain<true>(drain, 0, p.err, DEV_TIMEOUT_GEMM + 18);
    }
  } else {
    // ------------------------------------------------------------------ epilogue warps (both CTAs)
    const int q = warp & 3;
    const int r_in_tile = q * 32 + lane;
    const uint32_t leader_tempty = cluster_addr(tempty, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = cid; u < num_units; u += n_clusters) {
      int pm, nb, hh;
      decode(u, pm, nb, hh);
      const int row = pm * 2 * BM + (int)rank * BM + r_in_tile;
      const bool row_ok = row < p.M;
      if (EPI == EPI_GATED_RESIDUAL && row_ok) {
        const __nv_bfloat16* xr = p.resid + (size_t)row * p.ldr + nb * BN;
#pragma unroll
        for (int k = 0; k < BN / 64; ++k)
          if (nb * BN + k * 64 < p.N) asm volatile("prefetch.global.L2 [%0];" ::"l"(xr + k * 64));
      }
      if (!mbar_wait_warp<true>(&tfull[acc], acc_phase, abort_flag, p.err, DEV_TIMEOUT_GEMM + 17)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if (hh < 0)
        epilogue_tile<BN, EPI>(p, t_row, row, row_ok, nb);
      else  // a half tile: column block 2 nb + hh of width 128
        epilogue_tile<BN / 2, EPI>(p, t_row, row, row_ok, 2 * nb + hh);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(leader_tempty + acc * 8);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  cluster_sync();  // the pair's MMAs, commits and remote arrives are all done before either exits
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 2 * BN);
  }
}

constexpr long long kSkFixupKblocks = 64;

// Bytes of the arrival counters at the start of the stream-K scratch (then the partial slots):
// four per tail tile, and there are fewer than twice as many tail tiles as CTAs.
size_t sk_count_bytes(int grid) { return ((size_t)8 * grid * sizeof(int) + 1023) & ~(size_t)1023; }

// Stream-K plan of an M x N x K launch with num_sms SMs: returns the number of tail tiles (0: the
// plain schedule) and sets *grid.  With at least one full wave, the tail is the last full wave plus
// the remainder on all SMs; with fewer tiles than SMs, every tile, on twice as many CTAs (at most
// the SM count).  The fix-up of a split tile (its partial sums written, then read back and added
// by the last CTA, each at the memory latency of a loaded GPU) costs about as much time as 64
// k-blocks of the main loop, measured on the block's out and down projections; the tail is used
// only when it saves more k-blocks than that.
int sk_plan(int M, int N, int K, int num_sms, int bn, int* grid) {
  const int tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  const long long kb = K / BK;
  int g, sk;
  long long old_t, new_t;
  if (tiles >= num_sms) {
    const int full = tiles / num_sms, rem = tiles % num_sms;
    if (rem == 0) return 0;
    g = num_sms;
    sk = num_sms + rem;
    old_t = (full + 1) * kb;
    new_t = (full - 1) * kb + (sk * kb + g - 1) / g + 2;
  } else {
    g = 2 * tiles < num_sms ? 2 * tiles : num_sms;
    sk = tiles;
    old_t = kb;
    new_t = (sk * kb + g - 1) / g + 2;
  }
  if (old_t - new_t < kSkFixupKblocks) return 0;
  *grid = g;
  return sk;
}

template <int BN, int EPI>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a_in, int num_sms,
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
  GemmArgs a = a_in;
  const int num_m = (a.M + BM - 1) / BM;
  const int num_n = (EPI == EPI_SILU_GATE) ? (a.N / (BN / 2)) : (a.N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  int grid = tiles < num_sms ? tiles : num_sms;
  a.sk_tiles = 0;
  a.sk_count = nullptr;
  a.sk_partial = nullptr;
  if (kStreamK<EPI> && a.sk_scratch != nullptr) {
    int g = 0;
    const int t = sk_plan(a.M, a.N, a.K, num_sms, BN, &g);
    if (t > 0) {
      grid = g;
      a.sk_tiles = t;
      a.sk_count = static_cast<int*>(a.sk_scratch);
      a.sk_partial = reinterpret_cast<float*>(static_cast<uint8_t*>(a.sk_scratch) + sk_count_bytes(num_sms));
      e = cudaMemsetAsync(a.sk_count, 0, sk_count_bytes(num_sms), s);
      if (e != cudaSuccess) return e;
    }
  }
  // no programmatic launch after the counters' memset: it is not a kernel the launch could overlap
  return launch_kernel(kern, dim3(grid), dim3(kThreads), L::TOTAL, s, a.sk_tiles == 0, ta, tb, a);
}

// MI_GEMM_PAIRS=0 keeps every GEMM on the one-CTA kernel (for comparisons).
bool pair_disabled() {
  static const bool off = [] {
    const char* e = getenv("MI_GEMM_PAIRS");
    return e && e[0] == '0';
  }();
  return off;
}

// Clusters of two that can be resident at once with the pair kernel's shared memory (cached per
// device and epilogue); 0 when the query fails.
template <int EPI>
int pair_max_clusters(int num_sms) {
  static int cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    if (cudaFuncSetAttribute(gemm_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, PairSmem::TOTAL) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = PairSmem::TOTAL;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<EPI>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

template <int EPI>
cudaError_t launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a_in, int max_clusters,
                             cudaStream_t s) {
  GemmArgs a = a_in;
  const int num_pm = (a.M + 2 * BM - 1) / (2 * BM);
  const int num_n = (EPI == EPI_SILU_GATE) ? (a.N / 128) : (a.N + 255) / 256;
  const int tiles = num_pm * num_n;
  const int clusters = tiles < max_clusters ? tiles : max_clusters;
  // a partial last wave of at most half the clusters runs as half-width tiles on twice as many
  const int rem = tiles % clusters;
  a.half_from = (tiles > clusters && rem > 0 && 2 * rem <= clusters && (EPI != EPI_SILU_GATE || a.N % 128 == 0))
                    ? tiles - rem
                    : INT_MAX;
  return launch_kernel(gemm_pair_kernel<EPI>, dim3(2 * clusters), dim3(kThreads), PairSmem::TOTAL, s, true, ta, tb,
                       a);
}

// Launches the pair kernel may serve: more than one 128-row block and at least one full column tile.
bool pair_shape(int epi, int M, int N) {
  const bool wide = epi == EPI_SILU_GATE ? N >= 128 : N >= 256;
  return wide && M > BM && !pair_disabled();
}

// Whether a launch (given stream-K scratch) runs on the one-CTA kernel with a stream-K tail: the
// few-tile long-k launches (fewer of its tiles than SMs, whose k-blocks it spreads over up to twice
// as many CTAs) and tail launches the pair kernel cannot serve.  A launch with at least a wave of
// one-CTA tiles goes to the pair kernel instead, on its plain schedule: at 8260 x 3072 x 8192 (the
// guided step's down projection) and 16418 rows the pair kernel beats the one-CTA stream-K tail.
bool one_cta_tail(int epi, int M, int N, int K, int num_sms) {
  if (!(epi == EPI_STORE || epi == EPI_GATED_RESIDUAL || epi == EPI_STORE_F32)) return false;
  int g = 0;
  if (sk_plan(M, N, K, num_sms, 256, &g) == 0) return false;
  const int tiles = ((M + BM - 1) / BM) * ((N + 255) / 256);
  return tiles < num_sms || !pair_shape(epi, M, N);
}

// The pair kernel serves the launches of pair_shape() that do not take the one-CTA stream-K tail;
// the one-CTA kernel keeps the others (a single row block, the narrow velocity projection, the
// few-tile long-k launches).
template <int EPI>
cudaError_t launch_gemm_auto(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int num_sms,
                             cudaStream_t s) {
  const bool tail = a.sk_scratch != nullptr && one_cta_tail(EPI, a.M, a.N, a.K, num_sms);
  if (!tail && pair_shape(EPI, a.M, a.N)) {
    const int mc = pair_max_clusters<EPI>(num_sms);
    if (mc > 0) return launch_gemm_pair<EPI>(ta, tb, a, mc, s);
  }
  return launch_gemm<256, EPI>(ta, tb, a, num_sms, s);
}

}  // namespace

size_t gemm_sk_scratch_bytes(int epi, int M, int N, int K, int num_sms) {
  if (M <= 0 || N <= 0 || K <= 0 || num_sms <= 0 || !one_cta_tail(epi, M, N, K, num_sms)) return 0;
  return sk_count_bytes(num_sms) + (size_t)2 * num_sms * BM * 256 * sizeof(float);
}

cudaError_t gemm_launch(int epi, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int num_sms,
                        cudaStream_t s) {
  switch (epi) {
    case EPI_STORE:
      return launch_gemm_auto<EPI_STORE>(ta, tb, a, num_sms, s);
    case EPI_GATED_RESIDUAL:
      return launch_gemm_auto<EPI_GATED_RESIDUAL>(ta, tb, a, num_sms, s);
    case EPI_SILU_GATE:
      return launch_gemm_auto<EPI_SILU_GATE>(ta, tb, a, num_sms, s);
    case EPI_STORE_F32:
      return launch_gemm_auto<EPI_STORE_F32>(ta, tb, a, num_sms, s);
    case EPI_QKV_ROPE:
      return launch_gemm_auto<EPI_QKV_ROPE>(ta, tb, a, num_sms, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace mi
