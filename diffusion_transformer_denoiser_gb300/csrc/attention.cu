// Full (non-causal) attention at head dim 128 with an fp32 online softmax.
//
// The pages run the block's attention through a templated head-128 attention kernel with fp32
// softmax (MOSS-Image transformer on CUDA, "What it adds" and "Shared code").  This kernel is
// written for the 5th-generation tensor cores.  The unit of work is a pair of 128-row query tiles
// of one (batch, head); the keys are streamed once for both tiles.  The grid is persistent: one
// CTA per SM takes an equal share of all (unit, key tile) steps, a contiguous range cut into
// segments of one unit each, so no SM idles in a partial last wave.  A unit cut between two CTAs
// is finished by whichever part arrives second: the first writes its unnormalised O, running max
// and sum to scratch, the second adds both parts in a fixed order (keys from 0 first) and stores.
// Without scratch, or with more than 8 units per SM (where one CTA per unit balances better), the
// grid is one CTA per unit.
//   * warp 0   : TMA producer: the Q tiles of each segment, then K and V tiles of 128 keys into a
//                2-stage ring (K and V with their own barriers so a K slot frees as soon as both
//                score products have read it).  K comes from the packed [B, heads, S, 128] rows; V
//                is read in place from the QKV projection output through a strided 4-D map.
//   * warp 1   : issues (convergent warp, one elected lane per instruction), per key tile j, in this order
//                  O0 += P0 V_j,  S0 = Q0 K_{j+1}^T,  O1 += P1 V_j,  S1 = Q1 K_{j+1}^T
//                so the tensor core works on one query tile while the softmax works on the other.
//                Each P V is issued in two halves of 64 keys, each as soon as the softmax has
//                released that half of P.  A warp's MMA issue stalls while the tensor core's queue
//                is full and the issuer shares its SM sub-partition with two softmax warps, so its
//                loop carries nothing it can leave to others:
//   * warp 2   : wait proxy: waits for V of each key tile and K of the next and adds an arrival to
//                query tile 0's P barriers, which therefore imply those copies for the issuer.
//   * warp 3   : idle (it completes the first warpgroup, whose registers go to the softmax).
//   * warps 4-7 (query tile 0) and 8-11 (query tile 1): one thread per query row.  Scores come
//                from TMEM; the key tail and masked keys become -inf; the running max lives in
//                base 2 with log2(e)/sqrt(128) folded into one FMA (packed f32x2, as the row sum);
//                P is rounded to bf16 and written back into TMEM over the scores, where it is the A
//                operand of P V.  O is rescaled in TMEM only when a row's max grows by more than
//                2^8 (the stale max keeps every exponent <= 2^8, so P stays exact enough in bf16 and
//                the sum in fp32).  At a segment's end they normalise and store O (or write or
//                combine the parts of a cut unit) and release O for the next segment.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512); P_i = first 64
// columns of S_i.  tcgen05.mma operations of one thread execute in issue order, so S_i(j+1) may be
// issued right after the P_i(j) V_j product that still reads P_i(j) from the same columns.  Tile
// order, segment boundaries (a function of the shape and the SM count) and reduction order are
// fixed: results repeat bit for bit.
#include "mi_internal.h"
#include "ptx.cuh"

namespace mi {

namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int kThreads = 384;
// Register split: the launch gives every thread 168 registers (384 x 168 = 64512 of the SM's
// 65536).  The first warpgroup (producer, MMA issuer, two idle warps) drops to kRegsControl and
// the two softmax warpgroups rise to kRegsSoftmax, enough to hold a row's 128 scores with no
// spill: 128 x 104 + 256 x 200 = 64512, exactly the launch's pool.  The increase waits until
// the decrease has freed its registers, so the split must fit the pool the kernel was actually
// launched with; attention_launch checks that before the first launch.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 104;
constexpr int kRegsSoftmax = 200;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split exceeds the launch pool");
constexpr int TILE_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 tile = two 16 KB swizzled halves
constexpr int HALF_BYTES = TILE_BYTES / 2;

constexpr int OFF_Q = 0;                        // 2 query tiles
constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;   // 2 stages
constexpr int OFF_V = OFF_K + 2 * TILE_BYTES;   // 2 stages
constexpr int OFF_MASK = OFF_V + 2 * TILE_BYTES;
constexpr int kMaskWords = 2048;  // key-validity bitmask held in shared memory: up to 65536 keys
constexpr int OFF_BAR = OFF_MASK + kMaskWords * 4;
constexpr int OFF_SEG = OFF_BAR + 256;          // the CTA's segment list (int4 each) and its length
constexpr int SMEM_TOTAL = OFF_SEG + 16 * 16 + 16 + 1024;

constexpr uint32_t TM_S = 0;    // S_i at TM_S + 128 i (P_i in its first 64 columns)
constexpr uint32_t TM_O = 256;  // O_i at TM_O + 128 i
constexpr uint32_t TM_COLS = 512;
constexpr float kRescaleLog2 = 8.0f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

constexpr int kPartRowFloats = 130;                     // a row's 128 O values, then m and l
constexpr int kPartTileFloats = 128 * kPartRowFloats;   // one query tile of a part

// One CTA's share of the work: a contiguous range of (unit, key tile) steps, where unit
// u = (b * heads + h) * n_qp + qp is the pair of 128-row query tiles qp of one (batch, head).  The
// range is cut into segments of consecutive key tiles of one unit, listed once in shared memory
// ({u, first key tile, end key tile}) and walked by every role.  The launch keeps the list short:
// it splits units only while a CTA's share stays under kMaxSegs - 2 units.
constexpr int kMaxSegs = 16;

__device__ int build_segments(int4* tab, long long total, int n_kv) {
  long long w = total * blockIdx.x / gridDim.x;
  const long long w1 = total * (blockIdx.x + 1) / gridDim.x;
  int n = 0;
  while (w < w1 && n < kMaxSegs) {
    const int u = (int)(w / n_kv);
    const int jb = (int)(w % n_kv);
    const long long rem = w1 - w;
    const int je = (long long)(n_kv - jb) <= rem ? n_kv : jb + (int)rem;
    tab[n++] = make_int4(u, jb, je, 0);
    w += je - jb;
  }
  return n;
}

// 12 warps, 3 per SM sub-partition (16K registers each): 168 registers per thread at launch, which
// the launch bound below lets the compiler derive; the roles then trade registers as above.
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + OFF_Q;
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* v_full = bars + 3;    // [2]
  uint64_t* k_empty = bars + 5;   // [2]
  uint64_t* v_empty = bars + 7;   // [2]
  uint64_t* s_full = bars + 9;    // [2] per query tile
  uint64_t* p_full = bars + 11;   // [2][2] per query tile and half of P (keys 0-63, 64-127)
  uint64_t* o_done = bars + 15;   // [2] per query tile
  uint64_t* drain = bars + 17;
  uint64_t* q_empty = bars + 18;
  uint64_t* o_empty = bars + 19;  // [2] per query tile: its O has been read at the end of a segment
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 21);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* arrival = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2] per query tile

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.seq;
  const int n_kv = (S + BKV - 1) / BKV;
  const int n_qp = (S + 2 * BQ - 1) / (2 * BQ);
  int4* seg_tab = reinterpret_cast<int4*>(smem + OFF_SEG);
  volatile int* seg_count = reinterpret_cast<volatile int*>(smem + OFF_SEG + kMaxSegs * 16);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      // query tile 0's halves also count the wait proxy's arrival (V of the key tile, K of the next)
      mbar_init(&p_full[2 * i], i == 0 ? 5 : 4);
      mbar_init(&p_full[2 * i + 1], i == 0 ? 5 : 4);
      mbar_init(&o_done[i], 1);
      mbar_init(&o_empty[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *seg_count = build_segments(seg_tab, (long long)p.batch * p.n_heads * n_qp * n_kv, n_kv);
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
  grid_dep_wait();  // q, k and v are the previous kernel's outputs
  grid_dep_launch();

  // The two register regions are separate branches (warpgroup-uniform: every warp of a warpgroup
  // takes the same one), so the compiler holds each role to its own register budget.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------------------------ TMA producer
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        const int n_seg = *seg_count;
        int seg = 0;
        int kt = 0, k_issued = 0, v_issued = 0;
        bool ok = true;
        for (; ok && seg < n_seg;) {
          const int4 sg = seg_tab[seg];
          const int bh = sg.x / n_qp;
          const int b = bh / p.n_heads;
          const int h = bh % p.n_heads;
          const int q0 = (sg.x % n_qp) * (2 * BQ);
          // the previous segment's score products have read its Q
          if (seg > 0 && !mbar_wait(q_empty, (uint32_t)((seg - 1) & 1), abort_flag, p.err, DEV_TIMEOUT_ATTN + 1)) break;
          mbar_arrive_expect_tx(q_full, 2 * TILE_BYTES);
          tma_load_3d(sQ, &tmQ, q_full, 0, q0, bh);
          tma_load_3d(sQ + HALF_BYTES, &tmQ, q_full, 64, q0, bh);
          tma_load_3d(sQ + TILE_BYTES, &tmQ, q_full, 0, q0 + BQ, bh);
          tma_load_3d(sQ + TILE_BYTES + HALF_BYTES, &tmQ, q_full, 64, q0 + BQ, bh);
          ++seg;
          for (int j = sg.y; j < sg.z; ++j, ++kt) {
            const int st = (kt & 1);
            const uint32_t ph = (uint32_t)((kt >> 1) & 1);
            if (!mbar_wait(&k_empty[st], ph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ATTN + 1)) {
              ok = false;
              break;
            }
            uint8_t* k_dst = sK + st * TILE_BYTES;
            mbar_arrive_expect_tx(&k_full[st], TILE_BYTES);
            tma_load_3d(k_dst, &tmK, &k_full[st], 0, j * BKV, bh);
            tma_load_3d(k_dst + HALF_BYTES, &tmK, &k_full[st], 64, j * BKV, bh);
            k_issued = kt + 1;
            if (!mbar_wait(&v_empty[st], ph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_ATTN + 1)) {
              ok = false;
              break;
            }
            uint8_t* v_dst = sV + st * TILE_BYTES;
            mbar_arrive_expect_tx(&v_full[st], TILE_BYTES);
            tma_load_4d(v_dst, &tmV, &v_full[st], 0, h, j * BKV, b);
            tma_load_4d(v_dst + HALF_BYTES, &tmV, &v_full[st], 64, h, j * BKV, b);
            v_issued = kt + 1;
          }
        }
        // drain the copies still in flight (the last use of each barrier phase)
        if (seg > 0) mbar_wait_drain(q_full, (uint32_t)((seg - 1) & 1), p.err, DEV_TIMEOUT_ATTN + 2);
        for (int j = k_issued - 2 < 0 ? 0 : k_issued - 2; j < k_issued; ++j)
          mbar_wait_drain(&k_full[j & 1], (uint32_t)((j >> 1) & 1), p.err, DEV_TIMEOUT_ATTN + 2);
        for (int j = v_issued - 2 < 0 ? 0 : v_issued - 2; j < v_issued; ++j)
          mbar_wait_drain(&v_full[j & 1], (uint32_t)((j >> 1) & 1), p.err, DEV_TIMEOUT_ATTN + 2);
      }
    } else if (warp == 2) {
      // ------------------------------------------------------------------ wait proxy
      // Waits for V of each key tile and for K of the next one and adds an arrival to the matching
      // half of query tile 0's P barrier, so that the MMA issuer (whose every instruction sits on
      // the chain) needs no wait of its own for them: through these release/acquire pairs its wait
      // for P also orders the copies before its products.
      const int n_seg = *seg_count;
      int kt = 0;
      bool ok = true;
      for (int seg = 0; ok && seg < n_seg; ++seg) {
        const int n = seg_tab[seg].z - seg_tab[seg].y;
        for (int t = 0; t < n; ++t, ++kt) {
          // each arrival belongs to the phase of key tile kt: the previous phase of the barrier
          // must be complete first (the copies often land a key tile ahead of the softmax)
          const uint32_t prev = (uint32_t)((kt - 1) & 1);
          if ((kt > 0 && !mbar_wait_warp(&p_full[0], prev, abort_flag, p.err, DEV_TIMEOUT_ATTN + 9)) ||
              !mbar_wait_warp(&v_full[kt & 1], (uint32_t)((kt >> 1) & 1), abort_flag, p.err, DEV_TIMEOUT_ATTN + 9)) {
            ok = false;
            break;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[0]);
          if ((kt > 0 && !mbar_wait_warp(&p_full[1], prev, abort_flag, p.err, DEV_TIMEOUT_ATTN + 9)) ||
              (t + 1 < n &&
               !mbar_wait_warp(&k_full[(kt + 1) & 1], (uint32_t)(((kt + 1) >> 1) & 1), abort_flag, p.err,
                               DEV_TIMEOUT_ATTN + 9))) {
            ok = false;
            break;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[1]);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------------ MMA issuer
      // The whole warp runs this role convergently; each MMA and commit is issued by one elected lane.
      constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, 128, false, true);
      // operand descriptors of the two Q tiles and the two K and V stages, built once: the issuer
      // shares its SM sub-partition with two softmax warps, so every instruction off its loop counts
      const uint64_t qdesc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t qdesc1 = sdesc_sw128(smem_u32(sQ + TILE_BYTES), 16, 1024);
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t kdesc1 = sdesc_sw128(smem_u32(sK + TILE_BYTES), 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(sV), HALF_BYTES, 1024);
      const uint64_t vdesc1 = sdesc_sw128(smem_u32(sV + TILE_BYTES), HALF_BYTES, 1024);
      auto issue_s = [&](int i, int st) {  // S_i = Q_i K^T for the key tile in stage st
        const uint32_t d = tmem_base + TM_S + (uint32_t)i * 128u;
        const uint64_t qd = i ? qdesc1 : qdesc0;
        const uint64_t kd = st ? kdesc1 : kdesc0;
  #pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // the start-address field of a descriptor is in 16-byte units
          const uint32_t off = ((uint32_t)(kk >> 2) * HALF_BYTES + (uint32_t)(kk & 3) * 32u) >> 4;
          tc_mma_ss_warp(d, qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      // O_i (+)= P_i V over keys [64 half, 64 half + 64) of the key tile in stage st; the first
      // product of a segment starts O_i afresh
      auto issue_pv = [&](int i, int st, int half, bool first) {
        const uint32_t pa = tmem_base + TM_S + (uint32_t)i * 128u;
        const uint32_t d = tmem_base + TM_O + (uint32_t)i * 128u;
        const uint64_t vd = st ? vdesc1 : vdesc0;
  #pragma unroll
        for (int kk = 4 * half; kk < 4 * half + 4; ++kk) {
          // 16 keys per step: 8 packed P columns; V is MN-major (two 8-key groups 1024 B apart,
          // d halves 16 KB apart)
          tc_mma_ts_warp(d, pa + (uint32_t)kk * 8u, vd + (uint32_t)kk * (2048u >> 4), idesc_pv,
                         (!first || kk > 0) ? 1u : 0u);
        }
      };
      const int n_seg = *seg_count;
      int kt = 0;
      bool ok = true;
      for (int seg = 0; ok && seg < n_seg; ++seg) {
        const int n = seg_tab[seg].z - seg_tab[seg].y;
        const int kt0 = kt;
        ok = mbar_wait_warp(q_full, (uint32_t)(seg & 1), abort_flag, p.err, DEV_TIMEOUT_ATTN + 3) &&
             mbar_wait_warp(&k_full[kt0 & 1], (uint32_t)((kt0 >> 1) & 1), abort_flag, p.err, DEV_TIMEOUT_ATTN + 3);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, (kt0 & 1));
        tc_commit_warp(&s_full[0]);
        issue_s(1, (kt0 & 1));
        tc_commit_warp(&s_full[1]);
        tc_commit_warp(&k_empty[kt0 & 1]);
        if (n == 1) tc_commit_warp(q_empty);  // the segment's last score products are issued
        for (int t = 0; t < n; ++t) {
          kt = kt0 + t;
          const int st = (kt & 1);
          const uint32_t pp = (uint32_t)(kt & 1);
          const bool more = t + 1 < n;
          const int nst = ((kt + 1) & 1);
          const bool first = t == 0;
          // at a segment's first key tile, the previous segment's O has been read out
          if (first && seg > 0 &&
              !(mbar_wait_warp(&o_empty[0], (uint32_t)((seg - 1) & 1), abort_flag, p.err, DEV_TIMEOUT_ATTN + 4) &&
                mbar_wait_warp(&o_empty[1], (uint32_t)((seg - 1) & 1), abort_flag, p.err, DEV_TIMEOUT_ATTN + 4))) {
            ok = false;
            break;
          }
          // query tile 0: P V over the first 64 keys as soon as their half of P is in TMEM
          // (the first half of P_0 also implies that V of this key tile has landed: the wait proxy)
          if (!mbar_wait_warp(&p_full[0], pp, abort_flag, p.err, DEV_TIMEOUT_ATTN + 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(0, st, 0, first);
          if (!mbar_wait_warp(&p_full[1], pp, abort_flag, p.err, DEV_TIMEOUT_ATTN + 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(0, st, 1, first);
          tc_commit_warp(&o_done[0]);
          if (more) {  // the second half of P_0 implies that K of the next key tile has landed
            tc_fence_after();
            issue_s(0, nst);
            tc_commit_warp(&s_full[0]);
          }
          // query tile 1
          if (!mbar_wait_warp(&p_full[2], pp, abort_flag, p.err, DEV_TIMEOUT_ATTN + 6)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(1, st, 0, first);
          if (!mbar_wait_warp(&p_full[3], pp, abort_flag, p.err, DEV_TIMEOUT_ATTN + 6)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(1, st, 1, first);
          tc_commit_warp(&o_done[1]);
          tc_commit_warp(&v_empty[st]);
          if (more) {
            issue_s(1, nst);
            tc_commit_warp(&s_full[1]);
            tc_commit_warp(&k_empty[nst]);
            if (t + 2 == n) tc_commit_warp(q_empty);
          }
        }
        kt = kt0 + n;
      }
      tc_commit_warp(drain);
      mbar_wait_drain(drain, 0, p.err, DEV_TIMEOUT_ATTN + 7);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------------ softmax / epilogue
    const int wg = (warp - 4) >> 2;  // query tile of this warpgroup
    const int qw = warp & 3;         // TMEM lane quarter of this warp
    const int r = qw * 32 + lane;    // query row inside the tile == TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(qw * 32) << 16);
    const uint32_t t_s = t_lane + TM_S + (uint32_t)wg * 128u;
    const uint32_t t_o = t_lane + TM_O + (uint32_t)wg * 128u;
    const float sl2 = p.scale_log2;
    const int H = p.n_heads * kHeadDim;
    // key validity (tail and key mask) as a bitmask in shared memory, built by the 8 softmax warps
    // for the batch element of the current segment: bit k of word w says whether key 32 w + k may
    // be attended
    uint32_t* mask_words = reinterpret_cast<uint32_t*>(smem + OFF_MASK);
    const bool smem_mask = n_kv * 4 <= kMaskWords;
    int mask_b = -1;
    const int n_seg = *seg_count;
    int kt = 0;
    bool ok = true;
    for (int seg = 0; ok && seg < n_seg; ++seg) {
      const int b = seg_tab[seg].x / n_qp / p.n_heads;
      if (smem_mask && b != mask_b) {
        // both softmax warpgroups walk the same segments, so both reach this point for the same
        // batch element; the first barrier keeps a warpgroup still reading the old mask safe
        if (mask_b >= 0) asm volatile("bar.sync 1, 256;" ::: "memory");
        // warp w takes the 128-key chunks w, w + 8, ...; two chunks (8 byte loads per lane, all
        // independent, so their latencies overlap) per round
        const uint8_t* km = p.key_mask != nullptr ? p.key_mask + (size_t)b * S : nullptr;
        for (int c0 = warp - 4; c0 < n_kv; c0 += 16) {
          uint32_t v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int kc = (c0 + 8 * (i >> 2)) * 128 + (i & 3) * 32 + lane;
            v[i] = kc < S ? 1u : 0u;
            if (km != nullptr && kc < S) v[i] = km[kc];
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = c0 + 8 * (i >> 2);
            const uint32_t word = __ballot_sync(0xffffffffu, v[i] != 0);
            if (lane == 0 && c < n_kv) mask_words[c * 4 + (i & 3)] = word;
          }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");  // the 8 softmax warps only
        mask_b = b;
      }
      float m_run = neg_inf();  // reference max (base-2 units) the exponents are taken against
      float l_run = 0.0f;
      const int jb = seg_tab[seg].y;
      const int n = seg_tab[seg].z - jb;
      const int kt0 = kt;
      for (int t = 0; t < n; ++t) {
        kt = kt0 + t;
        const int j = jb + t;
        if (!mbar_wait_warp(&s_full[wg], (uint32_t)(kt & 1), abort_flag, p.err, DEV_TIMEOUT_ATTN + 8)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, sr + c * 32);
        tmem_ld_wait();
        const int kbase = j * BKV;
        uint32_t words[4];
        if (smem_mask) {
          const uint4 mw = *reinterpret_cast<const uint4*>(mask_words + j * 4);
          words[0] = mw.x;
          words[1] = mw.y;
          words[2] = mw.z;
          words[3] = mw.w;
        } else {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int kc = kbase + w * 32 + lane;
            bool valid = kc < S;
            if (valid && p.key_mask != nullptr) valid = p.key_mask[(size_t)b * S + kc] != 0;
            words[w] = __ballot_sync(0xffffffffu, valid);
          }
        }
        if ((words[0] & words[1] & words[2] & words[3]) != 0xffffffffu) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (!((words[c >> 5] >> (c & 31)) & 1u)) sr[c] = 0xff800000u;  // -inf
        }
        // row max and (below) row sum with 8 independent partials: short dependency chains
        float mp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mp[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int c = 8; c < 128; c += 8) {
#pragma unroll
          for (int k = 0; k < 8; ++k) mp[k] = fmaxf(mp[k], __uint_as_float(sr[c + k]));
        }
        const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        const float m_cand = mx * sl2;
        float alpha = 1.0f;
        const bool grow = m_cand > m_run + kRescaleLog2;  // also true for the first finite max
        if (grow) {
          alpha = ex2_approx(m_run - m_cand);
          m_run = m_cand;
        }
        const float m_use = (m_run == neg_inf()) ? 0.0f : m_run;
        if (t > 0) {
          // O_i holds the P V products of this segment up to the previous key tile, all complete:
          // the scores this warp waited for were issued after that product by the same thread,
          // and the tcgen05 operations of one thread complete in issue order.  It is rescaled
          // before the first half of the new P is released to the tensor core.
          if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              tmem_ld32(t_o + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(t_o + c * 32, o);
            }
          }
        }
        // packed f32x2 arithmetic (one instruction per pair of keys) for the exponent arguments
        // and the row sum: the softmax warps share each SM sub-partition with the MMA issuer or the
        // producer, and every issue slot they leave free shortens the issuer's path
        f32x2_t sp2[4] = {0ull, 0ull, 0ull, 0ull};
        const f32x2_t sl2x2 = f2_pack(sl2, sl2);
        const f32x2_t negm2 = f2_pack(-m_use, -m_use);
        // P in place, one half of the keys at a time: word c of sr receives the bf16 pair (2c,
        // 2c+1), whose scores were read at step c (ascending c never overwrites a score still to
        // be read).  Each half goes to TMEM over scores that are already in registers and is
        // released at once, so P V over keys 0-63 runs while keys 64-127 are exponentiated.
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
#pragma unroll
          for (int c = 32 * hp; c < 32 * hp + 32; ++c) {
            const f32x2_t z = f2_fma(f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sl2x2, negm2);
            float z0, z1;
            f2_unpack(z, z0, z1);
            const float e0 = ex2_approx(z0);
            const float e1 = ex2_approx(z1);
            sp2[c & 3] = f2_add(sp2[c & 3], f2_pack(e0, e1));
            sr[c] = pack_bf16x2(e0, e1);
          }
          tmem_st32(t_s + 32 * hp, sr + 32 * hp);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[2 * wg + hp]);
        }
        float sp[8];
        f2_unpack(sp2[0], sp[0], sp[1]);
        f2_unpack(sp2[1], sp[2], sp[3]);
        f2_unpack(sp2[2], sp[4], sp[5]);
        f2_unpack(sp2[3], sp[6], sp[7]);
        const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        l_run = l_run * alpha + sum;
      }
      kt = kt0 + n;
      if (!ok || !mbar_wait_warp(&o_done[wg], (uint32_t)((kt - 1) & 1), abort_flag, p.err, DEV_TIMEOUT_ATTN + 10)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int4 sg = seg_tab[seg];
      const int bh = sg.x / n_qp;
      const int h = bh % p.n_heads;
      const int row = (sg.x % n_qp) * (2 * BQ) + wg * BQ + r;
      __nv_bfloat16* dst_row = p.out + ((size_t)b * S + row) * H + (size_t)h * kHeadDim;
      if (sg.y == 0 && sg.z == n_kv) {
        // the whole unit: normalise and store
        const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
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
      } else {
        // part of a unit split between this CTA and a neighbour: the first part (keys from 0) is
        // the CTA's last segment, the second part its first.  The part goes to this CTA's scratch
        // slot (unnormalised O, laid out [32-column chunk][4-column group][row] so each warp store
        // covers 512 contiguous bytes, then m and l); the second of the two to arrive adds both,
        // in the fixed order first part + second part, and stores the normalised output.
        const bool first_part = sg.y == 0;
        float* mine = p.part + (((size_t)blockIdx.x * 2 + (first_part ? 1 : 0)) * 2 + wg) * kPartTileFloats;
        float* other = p.part + ((((size_t)blockIdx.x + (first_part ? 1 : -1)) * 2 + (first_part ? 0 : 1)) * 2 + wg) *
                                    kPartTileFloats;
        float4* mine4 = reinterpret_cast<float4*>(mine);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            __stcg(mine4 + (c * 8 + v) * 128 + r,
                   make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]), __uint_as_float(o[4 * v + 2]),
                               __uint_as_float(o[4 * v + 3])));
        }
        __stcg(mine + 128 * 128 + r, m_run);
        __stcg(mine + 128 * 128 + 128 + r, l_run);
        __threadfence();
        asm volatile("bar.sync %0, 128;" ::"r"(2 + wg) : "memory");
        if (qw == 0 && lane == 0) arrival[wg] = atomicAdd(p.count + 2 * sg.x + wg, 1);
        asm volatile("bar.sync %0, 128;" ::"r"(2 + wg) : "memory");
        if (arrival[wg] == 1) {
          __threadfence();
          const float m_o = __ldcg(other + 128 * 128 + r);
          const float l_o = __ldcg(other + 128 * 128 + 128 + r);
          const float mA = first_part ? m_run : m_o, lA = first_part ? l_run : l_o;
          const float mB = first_part ? m_o : m_run, lB = first_part ? l_o : l_run;
          const float M = fmaxf(mA, mB);
          const float wA = M == neg_inf() ? 0.0f : ex2_approx(mA - M);
          const float wB = M == neg_inf() ? 0.0f : ex2_approx(mB - M);
          const float l = fmaf(wA, lA, wB * lB);
          const float inv = l > 0.0f ? 1.0f / l : 0.0f;
          const float4* other4 = reinterpret_cast<const float4*>(other);
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float4 x[8];
#pragma unroll
            for (int v = 0; v < 8; ++v) x[v] = __ldcg(other4 + (c * 8 + v) * 128 + r);
            uint32_t o[32];
            tmem_ld32(t_o + c * 32, o);
            tmem_ld_wait();
            if (row < S) {
              float f[32];
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const float xo[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float own = __uint_as_float(o[4 * v + e]);
                  const float oA = first_part ? own : xo[e];
                  const float oB = first_part ? xo[e] : own;
                  f[4 * v + e] = fmaf(wA, oA, wB * oB) * inv;
                }
              }
              uint4* dst = reinterpret_cast<uint4*>(dst_row + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[v] = make_uint4(pack_bf16x2(f[v * 8 + 0], f[v * 8 + 1]), pack_bf16x2(f[v * 8 + 2], f[v * 8 + 3]),
                                    pack_bf16x2(f[v * 8 + 4], f[v * 8 + 5]), pack_bf16x2(f[v * 8 + 6], f[v * 8 + 7]));
            }
          }
          if (qw == 0 && lane == 0) p.count[2 * sg.x + wg] = 0;  // clean for the next launch
        }
      }
      // O_i has been read: the next segment's first P V may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[wg]);
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
                             const AttnArgs& a, int num_sms, cudaStream_t s) {
  static bool attr_done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    // the softmax warpgroups' register increase needs the pool the split was sized for
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_fwd_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < 128 * kRegsControl + 256 * kRegsSoftmax) return cudaErrorInvalidConfiguration;
    attr_done[dev] = true;
  }
  return launch_kernel(attn_fwd_kernel, dim3(attention_grid(a.batch, a.seq, a.n_heads, a.part != nullptr ? num_sms : 0)),
                       dim3(kThreads), SMEM_TOTAL, s, true, tq, tk, tv, a);
}

// Units are split between CTAs (one per SM) only while there are at most 8 units per SM.  With
// more, one CTA per unit wins: the partial last wave is a small share of the work, and the hardware
// hands the next unit to whichever SM frees up first, which absorbs the up to 10% spread in speed
// between SMs that a fixed share cannot (at 16418 rows, 10.3 units per SM, one CTA per unit takes
// 2.10 ms against 2.33 ms split; at 4130 rows, 2.7 units per SM, split takes 153 µs against 157).
static bool attention_splits(long long units, int num_sms) {
  static_assert(8 <= kMaxSegs - 3, "a CTA's share must fit the segment list");
  return num_sms > 0 && units > num_sms && units <= 8LL * num_sms;
}

int attention_grid(int batch, int seq, int n_heads, int num_sms) {
  const long long units = (long long)batch * n_heads * ((seq + 2 * BQ - 1) / (2 * BQ));
  return (int)(attention_splits(units, num_sms) ? num_sms : units);
}

size_t attention_scratch_bytes(int batch, int seq, int n_heads, int num_sms) {
  const long long units = (long long)batch * n_heads * ((seq + 2 * BQ - 1) / (2 * BQ));
  if (!attention_splits(units, num_sms)) return 0;
  return attention_count_bytes(batch, seq, n_heads) + (size_t)num_sms * 2 * 2 * kPartTileFloats * sizeof(float);
}

size_t attention_count_bytes(int batch, int seq, int n_heads) {
  const long long units = (long long)batch * n_heads * ((seq + 2 * BQ - 1) / (2 * BQ));
  return ((size_t)units * 2 * sizeof(int) + 255) & ~(size_t)255;
}

}  // namespace mi
