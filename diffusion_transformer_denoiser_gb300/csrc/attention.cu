// Full (non-causal) attention at head dim 128 with an fp32 online softmax.
//
// The pages run the block's attention through a templated head-128 attention kernel with fp32
// softmax (MOSS-Image transformer on CUDA, "What it adds" and "Shared code").  This kernel is
// written for the 5th-generation tensor cores.  One CTA owns 128 query rows of one (batch, head):
//   * warp 0   : TMA producer: the Q tile once, then K and V tiles of 128 keys into a 2-stage ring.
//                K comes from the packed [B, heads, S, 128] rows written by the q/k norm + rotary
//                kernel; V is read in place from the QKV projection output through a strided map.
//   * warp 1   : one thread issues S = Q K^T (M=128, N=128, K=128) into one of two TMEM score
//                buffers, and O += P V (B operand MN-major) into the TMEM output accumulator.
//   * warps 2-5: one thread per query row: scores from TMEM, key tail / key mask as -inf, running
//                max and sum in fp32 (base-2 with log2(e)/sqrt(128) folded in), P as bf16 into a
//                128-byte-swizzled shared tile, O rescaled in TMEM when the max moves, and the
//                final O / l written as bf16.
// S for tile j+1 is computed while the softmax works on tile j.  Tile order is fixed, so results
// repeat bit for bit.
#include "mi_internal.h"
#include "ptx.cuh"

namespace mi {

namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int kThreads = 192;
constexpr int TILE_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 tile = two 16 KB swizzled halves
constexpr int HALF_BYTES = TILE_BYTES / 2;

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;        // 2 stages
constexpr int OFF_V = OFF_K + 2 * TILE_BYTES;    // 2 stages
constexpr int OFF_P = OFF_V + 2 * TILE_BYTES;
constexpr int OFF_BAR = OFF_P + TILE_BYTES;
constexpr int SMEM_TOTAL = OFF_BAR + 256 + 1024;

constexpr uint32_t TM_S0 = 0;
constexpr uint32_t TM_O = 256;
constexpr uint32_t TM_COLS = 512;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + OFF_Q;
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sP = smem + OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* v_full = bars + 3;    // [2]
  uint64_t* kv_empty = bars + 5;  // [2]
  uint64_t* s_full = bars + 7;    // [2]
  uint64_t* s_empty = bars + 9;   // [2]
  uint64_t* p_full = bars + 11;
  uint64_t* o_ready = bars + 12;
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int S = p.seq;
  const int q0 = qt * BQ;
  const int n_kv = (S + BKV - 1) / BKV;
  const int bh = b * p.n_heads + h;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(o_ready, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, TILE_BYTES);
      tma_load_3d(sQ, &tmQ, q_full, 0, q0, bh);
      tma_load_3d(sQ + HALF_BYTES, &tmQ, q_full, 64, q0, bh);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1, abort_flag, p.err, DEV_TIMEOUT_ATTN + 1)) break;
        uint8_t* k_dst = sK + st * TILE_BYTES;
        uint8_t* v_dst = sV + st * TILE_BYTES;
        mbar_arrive_expect_tx(&k_full[st], TILE_BYTES);
        tma_load_3d(k_dst, &tmK, &k_full[st], 0, j * BKV, bh);
        tma_load_3d(k_dst + HALF_BYTES, &tmK, &k_full[st], 64, j * BKV, bh);
        mbar_arrive_expect_tx(&v_full[st], TILE_BYTES);
        tma_load_4d(v_dst, &tmV, &v_full[st], 0, h, j * BKV, b);
        tma_load_4d(v_dst + HALF_BYTES, &tmV, &v_full[st], 64, h, j * BKV, b);
        issued = j + 1;
      }
      // drain the copies still in flight: the last use of stage st is tile (issued-1 or issued-2)
      mbar_wait_drain(q_full, 0, p.err, DEV_TIMEOUT_ATTN + 2);
      for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j) {
        mbar_wait_drain(&k_full[j & 1], (j >> 1) & 1, p.err, DEV_TIMEOUT_ATTN + 2);
        mbar_wait_drain(&v_full[j & 1], (j >> 1) & 1, p.err, DEV_TIMEOUT_ATTN + 2);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, 128, false, true);
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t p_addr = smem_u32(sP);
      auto issue_qk = [&](int j) {
        const uint32_t k_addr = smem_u32(sK + (j & 1) * TILE_BYTES);
        const uint32_t d = tmem_base + TM_S0 + (uint32_t)(j & 1) * 128u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * HALF_BYTES + (uint32_t)(kk & 3) * 32u;
          tc_mma_ss(d, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024), idesc_qk,
                    kk > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.err, DEV_TIMEOUT_ATTN + 3) &&
                mbar_wait(&k_full[0], 0, abort_flag, p.err, DEV_TIMEOUT_ATTN + 3);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
        tc_commit(&s_full[0]);
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        if (j + 1 < n_kv) {
          const int nb = (j + 1) & 1;
          const uint32_t use = (uint32_t)((j + 1) >> 1);
          if (!mbar_wait(&s_empty[nb], (use & 1u) ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ATTN + 4) ||
              !mbar_wait(&k_full[nb], use & 1u, abort_flag, p.err, DEV_TIMEOUT_ATTN + 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_qk(j + 1);
          tc_commit(&s_full[nb]);
        }
        const int st = j & 1;
        if (!mbar_wait(p_full, j & 1, abort_flag, p.err, DEV_TIMEOUT_ATTN + 5) ||
            !mbar_wait(&v_full[st], (j >> 1) & 1, abort_flag, p.err, DEV_TIMEOUT_ATTN + 5)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sV + st * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a_off = (uint32_t)(kk >> 2) * HALF_BYTES + (uint32_t)(kk & 3) * 32u;
          // V is MN-major: 16 keys = two 8-row groups (SBO 1024); d halves 16 KB apart (LBO)
          tc_mma_ss(tmem_base + TM_O, sdesc_sw128(p_addr + a_off, 16, 1024),
                    sdesc_sw128(v_addr + (uint32_t)kk * 2048u, HALF_BYTES, 1024), idesc_pv,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&kv_empty[st]);
        tc_commit(o_ready);
      }
      tc_commit(drain);
      mbar_wait_drain(drain, 0, p.err, DEV_TIMEOUT_ATTN + 6);
    }
  } else {
    // ------------------------------------------------------------------ softmax / epilogue
    const int qw = warp & 3;
    const int r = qw * 32 + lane;  // query row inside the tile == TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(qw * 32) << 16);
    const float sl2 = p.scale_log2;
    float m_run = neg_inf();
    float l_run = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      if (!mbar_wait_warp(&s_full[sb], (j >> 1) & 1, abort_flag, p.err, DEV_TIMEOUT_ATTN + 7)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(t_lane + TM_S0 + sb * 128 + c * 32, sr + c * 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[sb]);

      float* s = reinterpret_cast<float*>(sr);
      const int kbase = j * BKV;
      if (p.key_mask != nullptr || kbase + BKV > S) {
        uint32_t words[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int kc = kbase + w * 32 + lane;
          bool valid = kc < S;
          if (valid && p.key_mask != nullptr) valid = p.key_mask[(size_t)b * S + kc] != 0;
          words[w] = __ballot_sync(0xffffffffu, valid);
        }
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (!((words[c >> 5] >> (c & 31)) & 1u)) s[c] = neg_inf();
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m_run, mx * sl2);
      const float m_use = (m_new == neg_inf()) ? 0.0f : m_new;
      const float alpha = ex2_approx(m_run - m_use);
      float sum = 0.0f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const float e = ex2_approx(fmaf(s[c], sl2, -m_use));
        s[c] = e;
        sum += e;
      }
      l_run = l_run * alpha + sum;
      m_run = m_new;

      if (j > 0) {
        // the previous P V product must be done before O is rescaled and P is overwritten
        if (!mbar_wait_warp(o_ready, (j - 1) & 1, abort_flag, p.err, DEV_TIMEOUT_ATTN + 8)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(t_lane + TM_O + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(t_lane + TM_O + c * 32, o);
          }
          tmem_st_wait();
        }
      }
      // P row -> swizzled K-major tile (two 64-key halves, 128 B per row, 16-B chunks XOR row%8)
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        const uint32_t off = (uint32_t)(c8 >> 3) * HALF_BYTES + (uint32_t)r * 128u +
                             ((uint32_t)((c8 & 7) ^ (r & 7)) << 4);
        uint4 v;
        v.x = pack_bf16x2(s[c8 * 8 + 0], s[c8 * 8 + 1]);
        v.y = pack_bf16x2(s[c8 * 8 + 2], s[c8 * 8 + 3]);
        v.z = pack_bf16x2(s[c8 * 8 + 4], s[c8 * 8 + 5]);
        v.w = pack_bf16x2(s[c8 * 8 + 6], s[c8 * 8 + 7]);
        *reinterpret_cast<uint4*>(sP + off) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && mbar_wait_warp(o_ready, (n_kv - 1) & 1, abort_flag, p.err, DEV_TIMEOUT_ATTN + 9)) {
      tc_fence_after();
      const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
      const int row = q0 + r;
      const int H = p.n_heads * kHeadDim;
      __nv_bfloat16* dst_row = p.out + ((size_t)b * S + row) * H + (size_t)h * kHeadDim;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(t_lane + TM_O + c * 32, o);
        tmem_ld_wait();
        if (row < S) {
          uint4* dst = reinterpret_cast<uint4*>(dst_row + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            dst[v] = make_uint4(
                pack_bf16x2(__uint_as_float(o[v * 8 + 0]) * inv, __uint_as_float(o[v * 8 + 1]) * inv),
                pack_bf16x2(__uint_as_float(o[v * 8 + 2]) * inv, __uint_as_float(o[v * 8 + 3]) * inv),
                pack_bf16x2(__uint_as_float(o[v * 8 + 4]) * inv, __uint_as_float(o[v * 8 + 5]) * inv),
                pack_bf16x2(__uint_as_float(o[v * 8 + 6]) * inv, __uint_as_float(o[v * 8 + 7]) * inv));
          }
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TM_COLS);
  }
}

}  // namespace

cudaError_t attention_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const AttnArgs& a, cudaStream_t s) {
  static bool attr_done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  dim3 grid((a.seq + BQ - 1) / BQ, a.n_heads, a.batch);
  attn_fwd_kernel<<<grid, kThreads, SMEM_TOTAL, s>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace mi
