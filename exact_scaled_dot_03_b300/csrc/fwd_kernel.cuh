// Exact attention forward (prefill / cross-attention) for sm_103a.
//
// What it computes: O = softmax(scale * Q K^T + causal mask) V and the row
// log-sum-exp, per (batch, query head), with GQA/MQA head sharing
// ([MG-A] §2.2-§2.4, §4.1; [PW] §2.1, §2.3). How: the score matrix is formed
// one 128x128 tile at a time in tensor memory and never leaves the SM; each
// query row keeps the running statistics of the blockwise softmax recurrence
// ([AUT] §8, its first two equations; [MG-A] §6.3): running max m, denominator
// l and the un-normalised sum u (held in TMEM), with o = u / l at the end.
//
// Sources: [MG-A] menggq.pages.dev "Transformer 架构的数学与计算深度解析";
// [AUT] auturnal.com "从注意力到 IO 感知执行" (v10); [PW] pwwt.cn news 6124947.
//
// CTA = two 128-row query tiles of one (batch, head) sharing every K/V tile.
//   warps 0-3 : softmax for query tile 0 (thread = one query row = one TMEM lane)
//   warps 4-7 : softmax for query tile 1
//   warp  8   : TMA producer (Q once, then the K/V ring)
//   warp  9   : TMEM allocator + issuer of the S = Q K^T MMAs
//   warp 10   : issuer of the O += P V MMAs
// Two issuers: every barrier wait of an issuing thread is a round trip of a
// few hundred cycles and every tcgen05.mma costs the thread tens of cycles,
// so one thread issuing everything cannot keep the tensor core fed; split,
// each waits only for its own inputs and their waits overlap.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D);
// the bf16 probabilities P_t are written over the first 64 columns of S_t and
// fed to the P.V MMA straight from TMEM.
//
// Head dim 64: O takes only 64 columns per tile, so P gets columns of its own
// (P0 [384,448), P1 [448,512)) instead of sharing S's. S_t can then be
// overwritten as soon as the softmax warps have read it: the MMA warp computes
// S of the next key tile while the softmax works on this one (one step ahead),
// and the softmax only waits for the previous P.V before storing the new P.
//
// Rescaling is lazy: the reference max m of a row only moves when the new
// tile's max exceeds it by more than 8 (in base-2 units). l and u always share
// the same reference, so o = u / l is unchanged in exact arithmetic; the
// exponentials stay <= 2^8, far from fp32/bf16 overflow.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "ptx.cuh"

namespace attn_dev {

struct FwdArgs {
  __nv_bfloat16* o;   // [B, Hq, Nq, D]
  float* lse;         // [B, Hq, Nq] natural-log LSE, or nullptr
  int B, Hq, Hkv, Nq, Nk;
  int group;          // Hq / Hkv
  int causal;
  int causal_offset;  // Nk - Nq: query i is aligned with key i + causal_offset
  int window;         // > 0: query i sees key j only if |j - (i + causal_offset)| < window
  int num_pairs;      // ceil(Nq / 256)
  float scale_log2;   // scale * log2(e)
  unsigned* status;   // library status word (see kStatus*)
  // RoPE ([PW] §5.3): when rope_cs is set, K has already been rotated and the
  // Q tiles are rotated in shared memory right after they land; rope_cs holds
  // (cos, sin) as [D/2 pairs][rope_T positions from rope_pmin]. Query i sits
  // at position i + causal_offset.
  const float2* rope_cs;
  int rope_pmin, rope_T;
  // Failure-detection test hook: when set, the softmax warps of query tile 0
  // of block (0, 0, 0) replace their first S wait by a wait on a barrier that
  // nothing arrives on, with a 1 ms limit (0 in normal use).
  int stall;
};

template <int D>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int BM = 128;                 // query rows per tile
  static constexpr int BN = 128;                 // keys per K/V tile
  static constexpr int KBLK = D / 64;            // 64-column (128-byte) swizzle blocks per row
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int BLOCK_BYTES = 128 * 64 * 2;     // one 128-row x 64-col swizzle block
  static constexpr int TILE_BYTES = KBLK * BLOCK_BYTES;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + STAGES * TILE_BYTES;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2], pv_done[2], drain,
  // q_ready, stall, s_free[2]
  static constexpr int NUM_BARS = 1 + 4 * STAGES + 11;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + tmem base/abort words + alignment slack
  static constexpr int THREADS = 352;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 256;
  static constexpr bool SEP_P = (D == 64);       // P in columns of its own (see the header comment)
  static constexpr uint32_t P_COL = 384;         // SEP_P only
};

// Wait sites (recorded in status[1] when a bounded wait gives up).
enum : unsigned {
  kSiteQFull = 1, kSiteKEmpty, kSiteVEmpty, kSiteKFull, kSiteVFull, kSitePvDoneMma, kSitePFull,
  kSiteSFull, kSitePvDoneRescale, kSitePvDoneEpi, kSiteDrain, kSiteLoadDrain
};

// Keys query row r sees: [lo, hi] (empty if hi < lo). Causal: keys up to the
// aligned one; local window: within window - 1 of it on either side
// ([IMR] masking section; [AUT] §2 Longformer; [PW] §6.1).
template <bool WIN>
__device__ __forceinline__ void fwd_row_keys(const FwdArgs& a, long long r, int& lo, int& hi) {
  const long long dg = r + a.causal_offset;
  long long l = 0, h = (long long)a.Nk - 1;
  if (WIN) {
    l = max(l, dg - a.window + 1);
    h = min(h, dg + a.window - 1);
  }
  if (a.causal) h = min(h, dg);
  lo = (int)min(l, (long long)a.Nk);
  hi = (int)max(h, -1LL);
}

// The 128-key tiles [jb, je) a 128-row query tile starting at row r0 must
// visit (both ends move forward with r0, so the rows' ranges are covered by
// [lo(first row), hi(last row)]).
template <bool WIN>
__device__ __forceinline__ void fwd_kv_tiles(const FwdArgs& a, int r0, int& jb, int& je) {
  jb = je = 0;
  if (r0 >= a.Nq) return;
  int lo, hi, lo2, hi2;
  fwd_row_keys<WIN>(a, r0, lo, hi);
  fwd_row_keys<WIN>(a, min(r0 + 127, a.Nq - 1), lo2, hi2);
  if (hi2 < lo) return;
  jb = WIN ? lo / 128 : 0;  // without a window every query tile starts at key 0
  je = hi2 / 128 + 1;
}

// WIN: a local window is in force (the windowless instance keeps every range
// offset a compile-time zero).
template <int D, bool WIN>
__global__ void __launch_bounds__(352, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + C::STAGES;
  uint64_t* v_full = k_empty + C::STAGES;
  uint64_t* v_empty = v_full + C::STAGES;
  uint64_t* s_full = v_empty + C::STAGES;  // [2]
  uint64_t* p_full = s_full + 2;           // [2]
  uint64_t* pv_done = p_full + 2;          // [2]
  uint64_t* drain = pv_done + 2;
  uint64_t* q_ready = drain + 1;  // RoPE only: both Q tiles rotated in shared memory
  uint64_t* stall_bar = q_ready + 1;  // test hook only: never arrived on
  uint64_t* s_free = stall_bar + 1;   // [2] head dim 64: S_t read into registers
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int pair = a.num_pairs - 1 - blockIdx.y;  // heaviest (latest) causal rows first
  const int b = blockIdx.z;
  const int hkv = h / a.group;
  const int q_base = pair * 256;
  // Key tiles of query tile t: [jb[t], jb[t] + n_kv[t]); the CTA streams
  // [j0, j0 + n_kv_max) of them, K/V stage = stream position % STAGES.
  int jb[2], je[2], n_kv[2];
  fwd_kv_tiles<WIN>(a, q_base, jb[0], je[0]);
  fwd_kv_tiles<WIN>(a, q_base + 128, jb[1], je[1]);
  n_kv[0] = je[0] - jb[0];
  n_kv[1] = je[1] - jb[1];
  const int j0 = !WIN ? 0 : n_kv[0] > 0 ? (n_kv[1] > 0 ? min(jb[0], jb[1]) : jb[0]) : jb[1];
  const int n_kv_max = (n_kv[0] > 0 || n_kv[1] > 0)
                           ? max(n_kv[0] > 0 ? je[0] : 0, n_kv[1] > 0 ? je[1] : 0) - j0 : 0;
  auto uses = [&](int t, int j) { return j >= jb[t] && j < je[t]; };  // query tile t visits key tile j

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full + t, 1);
      mbar_init(p_full + t, 128);
      mbar_init(pv_done + t, 1);
      mbar_init(s_free + t, 128);
    }
    mbar_init(drain, 2);  // one commit from each MMA issuer
    mbar_init(q_ready, 256);
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_kv_max > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t qbytes = 0;
      for (int t = 0; t < 2; ++t) qbytes += n_kv[t] > 0 ? C::TILE_BYTES : 0;
      mbar_arrive_expect_tx(q_full, qbytes);
      const uint64_t stream_once = l2_policy_evict_first();  // Q is read by this CTA only
      for (int t = 0; t < 2; ++t) {
        if (n_kv[t] == 0) continue;
        for (int kb = 0; kb < C::KBLK; ++kb)
          tma_load_3d_hint(sQ + t * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tm_q, q_full, kb * 64, q_base + 128 * t,
                           b * a.Hq + h, stream_once);
      }
      int k_issued = 0, v_issued = 0;  // K and V tiles whose copies were started
      for (int js = 0; js < n_kv_max; ++js) {
        const int j = j0 + js;  // key tile
        const int s = js % C::STAGES;
        const int u = js / C::STAGES;
        if (u > 0 && !mbar_wait(k_empty + s, (u - 1) & 1, a.status, kSiteKEmpty, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(k_full + s, C::TILE_BYTES);
        for (int kb = 0; kb < C::KBLK; ++kb)
          tma_load_3d(sK + s * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tm_k, k_full + s, kb * 64, j * 128,
                      b * a.Hkv + hkv);
        k_issued = js + 1;
        if (u > 0 && !mbar_wait(v_empty + s, (u - 1) & 1, a.status, kSiteVEmpty, abort_flag)) {
          *abort_flag = 1;  // K of this tile is in flight, V is not
          break;
        }
        mbar_arrive_expect_tx(v_full + s, C::TILE_BYTES);
        for (int kb = 0; kb < C::KBLK; ++kb)
          tma_load_3d(sV + s * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tm_v, v_full + s, kb * 64, j * 128,
                      b * a.Hkv + hkv);
        v_issued = js + 1;
        if (*abort_flag) break;
      }
      if (*abort_flag) {
        // Let every copy still in flight land before the CTA exits: the last
        // STAGES copies started into each ring (earlier ones were consumed).
        mbar_wait(q_full, 0, a.status, kSiteLoadDrain);
        for (int js = max(0, k_issued - C::STAGES); js < k_issued; ++js)
          mbar_wait(k_full + js % C::STAGES, (js / C::STAGES) & 1, a.status, kSiteLoadDrain);
        for (int js = max(0, v_issued - C::STAGES); js < v_issued; ++js)
          mbar_wait(v_full + js % C::STAGES, (js / C::STAGES) & 1, a.status, kSiteLoadDrain);
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // Each descriptor is a precomputed low word plus a compile-time offset
    // (see sw128_desc_lo), which keeps the issuing thread's own instructions few.
    if (lane == 0 && n_kv_max > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      constexpr uint32_t kHi = sw128_desc_hi(1024);            // 8-row atoms 1024 bytes apart
      constexpr uint32_t kTileW = C::TILE_BYTES >> 4;          // one tile, in descriptor address units
      bool ok = true;
      if (warp == 9) {
        // S_t = Q_t K^T for every key tile, over head-dim steps of 16
        const uint32_t q_lo = sw128_desc_lo(smem_u32(sQ), 16);  // K-major Q and K
        const uint32_t k_lo = sw128_desc_lo(smem_u32(sK), 16);
        ok = mbar_wait(a.rope_cs != nullptr ? q_ready : q_full, 0, a.status, kSiteQFull, abort_flag);
        for (int js = 0; ok && js < n_kv_max; ++js) {
          const int j = j0 + js;  // key tile; query tile t is at its step j - jb[t]
          const int s = js % C::STAGES;
          if (!(ok = mbar_wait(k_full + s, (js / C::STAGES) & 1, a.status, kSiteKFull, abort_flag))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok || !uses(t, j)) continue;
            if (j > jb[t]) {
              // S_t is overwritten: with P aliased on S the previous P.V must be done,
              // with P in columns of its own the softmax must have read the previous S.
              if constexpr (C::SEP_P)
                ok = mbar_wait(s_free + t, (j - jb[t] - 1) & 1, a.status, kSitePvDoneMma, abort_flag);
              else
                ok = mbar_wait(pv_done + t, (j - jb[t] - 1) & 1, a.status, kSitePvDoneMma, abort_flag);
              if (!ok) break;
              tc_fence_after_sync();
            }
            const uint32_t a0 = q_lo + t * kTileW, b0 = k_lo + s * kTileW;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = static_cast<uint32_t>(((kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32) >> 4);
              umma_ss_w(tmem + 128 * t, a0 + off, kHi, b0 + off, kHi, idesc_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full + t);
          }
          if (!ok) break;
          umma_commit(k_empty + s);
        }
      } else {
        // O_t += P_t V for every key tile, over key steps of 16; P_t is read from TMEM
        const uint32_t v_lo = sw128_desc_lo(smem_u32(sV), C::BLOCK_BYTES);  // MN-major V
        for (int js = 0; ok && js < n_kv_max; ++js) {
          const int j = j0 + js;
          const int s = js % C::STAGES;
          if (!(ok = mbar_wait(v_full + s, (js / C::STAGES) & 1, a.status, kSiteVFull, abort_flag))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok || !uses(t, j)) continue;
            if (!(ok = mbar_wait(p_full + t, (j - jb[t]) & 1, a.status, kSitePFull, abort_flag))) break;
            tc_fence_after_sync();
            const uint32_t p_col = C::SEP_P ? C::P_COL + 64 * t : 128 * t;
            const uint32_t b0 = v_lo + s * kTileW;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_ts_w(tmem + C::O_COL + D * t, tmem + p_col + kk * 8, b0 + kk * (16 * 128 >> 4), kHi, idesc_pv,
                        (j > jb[t] || kk > 0) ? 1u : 0u);
            umma_commit(pv_done + t);
          }
          if (!ok) break;
          umma_commit(v_empty + s);
        }
      }
      if (!ok) *abort_flag = 1;
      // Every MMA either issuer started has finished before TMEM is released
      // (the barrier completes once both have committed).
      umma_commit(drain);
      mbar_wait(drain, 0, a.status, kSiteDrain);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = q_base + 128 * t + wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + 128 * t;
    const uint32_t tO = tmem + lane_off + C::O_COL + D * t;
    const uint32_t tP = C::SEP_P ? tmem + lane_off + C::P_COL + 64 * t : tS;  // where P is stored
    const int nk = t == 0 ? n_kv[0] : n_kv[1];   // selects, not a dynamic index (keeps them in registers)
    const int jb_t = t == 0 ? jb[0] : jb[1];
    const float sl2 = a.scale_log2;
    // keys this row sees: [vis_lo, vis_hi]; a key tile needs per-element masking
    // when it crosses the left edge of the tile's last row or the right edge
    // of its first row (the edges only move forward with the row)
    int vis_lo, vis_hi, lo_last, hi_first, unused;
    fwd_row_keys<WIN>(a, row, vis_lo, vis_hi);
    fwd_row_keys<WIN>(a, min(q_base + 128 * t + 127, max(a.Nq - 1, 0)), lo_last, unused);
    fwd_row_keys<WIN>(a, q_base + 128 * t, unused, hi_first);
    float m_used = -CUDART_INF_F;  // reference max, base-2 scaled units
    float l = 0.f;
    bool ok = true;
    if (a.rope_cs != nullptr) {
      // RoPE on this thread's Q row, in place in the swizzled tile: pair p of
      // chunk c (8 components) is the 32-bit word p of the chunk.
      if (nk > 0 && row < a.Nq) {
        // The row's (cos, sin) pairs are fetched before Q lands, so the loads
        // overlap the Q copy instead of following it; the table is pair-major,
        // so the warp's 32 consecutive rows read 256 contiguous bytes per pair.
        const float2* tab = a.rope_cs + (row + a.causal_offset - a.rope_pmin);
        float2 cs[D / 2];
#pragma unroll
        for (int i = 0; i < D / 2; ++i) cs[i] = __ldg(tab + (size_t)i * a.rope_T);
        if (!(ok = mbar_wait(q_full, 0, a.status, kSiteQFull, abort_flag))) *abort_flag = 1;
        const int rloc = wq * 32 + lane;
        uint8_t* qrow = sQ + t * C::TILE_BYTES + rloc * 128;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          uint4* p = reinterpret_cast<uint4*>(qrow + (c >> 3) * C::BLOCK_BYTES + (((c & 7) ^ (rloc & 7)) << 4));
          const uint4 w = *p;
          uint32_t in[4] = {w.x, w.y, w.z, w.w}, out[4];
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            const float x = __uint_as_float(in[k2] << 16), y = __uint_as_float(in[k2] & 0xffff0000u);
            const float2 t2 = cs[4 * c + k2];
            out[k2] = pack_bf16x2(x * t2.x - y * t2.y, x * t2.y + y * t2.x);
          }
          if (ok) *p = make_uint4(out[0], out[1], out[2], out[3]);
        }
        fence_proxy_async_smem();  // the MMA reads Q through the async proxy
      }
      mbar_arrive(q_ready);
    }
    // test hook: the first S wait of query tile 0 in block (0, 0, 0) stalls
    const bool stall = a.stall != 0 && t == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
    for (int j = 0; ok && j < nk; ++j) {  // step j visits key tile jb[t] + j
      if (stall) {  // gives up after 1 ms (nothing arrives), then takes the abort path
        mbar_wait(stall_bar, 0, a.status, kSiteSFull, abort_flag, kStallLimitNs);
        ok = false;
        break;
      }
      if (!(ok = mbar_wait(s_full + t, j & 1, a.status, kSiteSFull, abort_flag))) break;
      tc_fence_after_sync();
      float sv[128];
      {
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_reg_fence(sr[c]);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[32 * c + i] = __uint_as_float(sr[c][i]);
        }
      }
      if constexpr (C::SEP_P) {  // S_t is in registers: the MMA warp may compute the next one into it
        tc_fence_before_sync();
        mbar_arrive(s_free + t);
      }
      const int key0 = (jb_t + j) * 128;
      if (key0 + 127 > hi_first || (WIN && key0 < lo_last)) {  // tile-uniform: an edge crosses the tile
        const int rel_lo = vis_lo - key0, rel_hi = vis_hi - key0;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          sv[c] = ((WIN && c < rel_lo) || c > rel_hi) ? -CUDART_INF_F : sv[c];
      }
      // Row max with three-input max (half the instructions of a pairwise
      // chain; four independent chains for latency).
      float mx0 = fmax3(sv[0], sv[1], sv[2]), mx1 = fmax3(sv[3], sv[4], sv[5]);
      float mx2 = fmax3(sv[6], sv[7], sv[8]), mx3 = fmax3(sv[9], sv[10], sv[11]);
#pragma unroll
      for (int c = 12; c + 8 <= 128; c += 8) {
        mx0 = fmax3(mx0, sv[c], sv[c + 1]);
        mx1 = fmax3(mx1, sv[c + 2], sv[c + 3]);
        mx2 = fmax3(mx2, sv[c + 4], sv[c + 5]);
        mx3 = fmax3(mx3, sv[c + 6], sv[c + 7]);
      }
      mx0 = fmax3(mx0, sv[124], sv[125]);
      mx1 = fmax3(mx1, sv[126], sv[127]);
      const float m_new = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      const bool need = m_new > m_used + 8.0f;
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_used - m_new);  // 0 when m_used is still -inf
        m_used = m_new;
        l *= alpha;
      }
      // p = 2^(s * scale * log2(e) - m), packed to bf16 pairs over the first
      // 64 columns of S (the scores are dead once read into registers).
      const float m_ref = (m_used == -CUDART_INF_F) ? 0.f : m_used;
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = 64 * half + 2 * i;
          float x0, x1;
          fma2(x0, x1, sv[c], sv[c + 1], sl2, sl2, -m_ref, -m_ref);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          add2(l0, l1, p0, p1);
          pk[i] = pack_bf16x2(p0, p1);
        }
        if (C::SEP_P && half == 0 && j > 0) {
          // P_t's columns are free once the previous P.V has read them.
          ok = mbar_wait(pv_done + t, (j - 1) & 1, a.status, kSitePvDoneRescale, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform: the TMEM stores below are warp-collective
            ok = false;
            break;
          }
          tc_fence_after_sync();
        }
        tmem_st32(tP + 32 * half, pk);
      }
      if (!ok) break;
      l += l0 + l1;
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // Bring the accumulated u onto the new reference before P.V adds to it.
        if (!(ok = mbar_wait(pv_done + t, (j - 1) & 1, a.status, kSitePvDoneRescale, abort_flag))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(tO + 32 * c, orr);
          tmem_wait_ld();
          tmem_reg_fence(orr);
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
          tmem_st32(tO + 32 * c, orr);
        }
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(p_full + t);
    }
    if (!ok) *abort_flag = 1;
    // ---------------------------------------------------------- epilogue
    bool have_o = false;
    if (ok && nk > 0) {
      ok = mbar_wait(pv_done + t, (nk - 1) & 1, a.status, kSitePvDoneEpi, abort_flag);
      tc_fence_after_sync();
      have_o = ok;
    }
    have_o = __all_sync(0xffffffffu, have_o);  // guards warp-collective TMEM loads
    const bool in_range = row < a.Nq;
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const uint64_t out_policy = l2_policy_evict_first();
    __nv_bfloat16* orow = a.o + ((size_t)(b * a.Hq + h) * a.Nq + (in_range ? row : 0)) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t orr[32];
      if (have_o) {
        tmem_ld32(tO + 32 * c, orr);
        tmem_wait_ld();
        tmem_reg_fence(orr);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) orr[i] = 0u;
      }
      uint32_t packed[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        packed[i] = pack_bf16x2(__uint_as_float(orr[2 * i]) * inv_l, __uint_as_float(orr[2 * i + 1]) * inv_l);
      if (in_range) {
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i)  // O is written once: evict-first keeps K/V of other CTAs in L2
          st_global_v4_hint(dst + i, make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]),
                            out_policy);
      }
    }
    if (a.lse != nullptr && in_range) {
      a.lse[(size_t)(b * a.Hq + h) * a.Nq + row] =
          l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace attn_dev
