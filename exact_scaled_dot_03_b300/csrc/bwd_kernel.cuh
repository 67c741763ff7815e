// Exact attention backward for sm_103a: dQ, dK, dV of
// O = softmax(scale * Q K^T + causal mask) V, with the scores recomputed from
// Q, K and the forward's row log-sum-exp instead of being stored ([MG-A] §3.3
// says standard attention keeps the N x N matrix for the backward pass;
// [MG-B] §3.2, engineering results: the tiled method recomputes it).
//
// The gradients are the chain rule through the forward definition:
//   P = exp(S - lse), dV = P^T dO, dP = dO V^T, dS = P * (dP - Dl),
//   Dl_i = sum_t dO_it O_it (equal to sum_j P_ij dP_ij), dQ = scale dS K,
//   dK = scale dS^T Q; the query heads of a GQA group add into one dK, dV.
//
// Sources: [MG-A] menggq.pages.dev "Transformer 架构的数学与计算深度解析";
// [MG-B] menggq.pages.dev "Transformer 深度进阶：从矩阵视角到 FlashAttention 工程优化".
//
// Three kernels, no atomics (the result is deterministic):
//   bwd_prep_kernel      per query row: lse * log2 e and Dl (two arrays), each
//                        head padded to a multiple of 128 rows with +inf and 0
//                        so that padded rows get P = 0.
//   attn_bwd_dkdv_kernel CTA = one 128-key tile of one (batch, KV head). It
//                        streams every query tile of every query head of the
//                        group; dK and dV accumulate in TMEM.
//   attn_bwd_dq_kernel   CTA = one 128-row query tile; streams its key tiles;
//                        dQ accumulates in TMEM.
// Both main kernels: warps 0-7 elementwise (two warpgroups, each owning half
// g of the 128 columns of a score tile; thread = TMEM lane = row), warp 8 TMA
// producer, warp 9 TMEM allocator + issuer of the score-shaped MMAs (S^T and
// dP^T, or S and dP), warp 10 issuer of the accumulating MMAs (dV and dK, or
// dQ): a barrier wait costs an issuing thread a round trip of a few hundred
// cycles, so two issuers whose waits overlap keep the tensor core fed where
// one could not. The elementwise work
// of a step runs in two phases, P = exp2(S - lse) (the exponentials) as soon
// as S is in TMEM and dS = P (dP - Dl) once dP is, so each phase overlaps a
// different MMA group (all MMAs are M = N = 128). In the dK/dV kernel, where
// lse and Dl belong to the columns, one extra K=16 MMA (a tile of ones times
// the column values split into three bf16 parts) seeds S^T with -lse/scale and
// dP^T with -Dl, so the elementwise warps load no per-column value:
//   dK/dV step: S^T | dP^T (P phase) | dV (dS phase) | dK
//   dQ step:    S(n+1) (as soon as S(n) is in registers) | dP(n+1) (while dS(n) and dQ(n) run) | dQ(n)
// (dP double-buffered in the dQ kernel, so dP(n+1) waits only for dQ(n-1)).
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "ptx.cuh"

namespace attn_dev {

struct BwdArgs {
  __nv_bfloat16* dq;   // [B, Hq, Nq, D]
  __nv_bfloat16* dk;   // [B, Hkv, Nk, D]
  __nv_bfloat16* dv;   // [B, Hkv, Nk, D]
  const float* lse2;   // [B * Hq][Nq_pad]: lse * log2 e; padded rows +inf
  const float* dl;     // [B * Hq][Nq_pad]: Dl = sum_t dO_t O_t; padded rows 0
  // Per 128-row query tile, the K=16 B operands that seed the dK/dV kernel's
  // accumulators (layout: bwd_seed_offset): -lse/scale and -Dl, each split
  // into three bf16 parts (columns 0-2; 3-15 zero). 4 KiB per tile and array.
  const uint8_t* seed_l;
  const uint8_t* seed_d;
  int B, Hq, Hkv, Nq, Nk, Nq_pad;
  int group;           // Hq / Hkv
  int causal;
  int causal_offset;   // Nk - Nq: query i is aligned with key i + causal_offset
  float scale;         // applied to dQ and dK in the epilogues
  float scale_log2;    // scale * log2(e)
  unsigned* status;
  // Failure-detection test hook: when set, the elementwise warpgroup 0 of the
  // dK/dV kernel's block (0, 0, 0) replaces its first score wait by a wait on
  // a barrier that nothing arrives on, with a 1 ms limit (0 in normal use).
  int stall;
};

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int KBLK = D / 64;
  static constexpr int BLOCK_BYTES = 128 * 64 * 2;   // 128 rows x 64 columns, 128-byte swizzle
  static constexpr int TILE_BYTES = KBLK * BLOCK_BYTES;
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int SEED_BYTES = 128 * 16 * 2;    // one 128 x 16 bf16 seed operand
  static constexpr int THREADS = 352;
  static constexpr uint32_t TMEM_COLS = 512;

  // dK/dV kernel: K, V once; Q, dO and (lse2, Dl) per stage.
  static constexpr int KV_K_OFF = 0;
  static constexpr int KV_V_OFF = TILE_BYTES;
  static constexpr int KV_Q_OFF = 2 * TILE_BYTES;
  static constexpr int KV_DO_OFF = KV_Q_OFF + STAGES * TILE_BYTES;
  static constexpr int KV_SEED_OFF = KV_DO_OFF + STAGES * TILE_BYTES;      // per stage: -lse seed, -Dl seed
  static constexpr int KV_ONES_OFF = KV_SEED_OFF + STAGES * 2 * SEED_BYTES;  // 128 x 16: ones in columns 0-2
  static constexpr int KV_BAR_OFF = KV_ONES_OFF + SEED_BYTES;
  // kv_full, full[S], empty[S], s_full, dp_full, p_full[2], ds_full[2], dv_done, dk_done, acc_done, drain, stall
  static constexpr int KV_NUM_BARS = 1 + 2 * STAGES + 11;
  static constexpr int KV_MISC_OFF = KV_BAR_OFF + KV_NUM_BARS * 8;
  static constexpr int KV_SMEM_BYTES = KV_MISC_OFF + 16 + 1024;
  // TMEM columns: S^T, dP^T (128 each; P^T and dS^T are written back over
  // them as packed bf16), then the dV and dK accumulators.
  static constexpr uint32_t T_ST = 0, T_DPT = 128, T_DV = 256, T_DK = 256 + D;

  // dQ kernel: Q, dO once; K, V per stage.
  static constexpr int Q_Q_OFF = 0;
  static constexpr int Q_DO_OFF = TILE_BYTES;
  static constexpr int Q_K_OFF = 2 * TILE_BYTES;
  static constexpr int Q_V_OFF = Q_K_OFF + STAGES * TILE_BYTES;
  static constexpr int Q_BAR_OFF = Q_V_OFF + STAGES * TILE_BYTES;
  // q_full, full[S], empty[S], s_full, s_free, dp_full[2] (per dP buffer), ds_full[2][2] (per dP
  // buffer and warpgroup), dq_done[2] (per dP buffer), acc_done, drain
  static constexpr int Q_NUM_BARS = 1 + 2 * STAGES + 13;
  static constexpr int Q_MISC_OFF = Q_BAR_OFF + Q_NUM_BARS * 8;
  static constexpr int Q_SMEM_BYTES = Q_MISC_OFF + 16 + 1024;
  // TMEM columns: S, dP buffer 0 (dS written back over it), dQ, dP buffer 1.
  static constexpr uint32_t T_S = 0, T_DP0 = 128, T_DQ = 256, T_DP1 = 384;
};

// Wait sites recorded in status[1] by the backward kernels.
enum : unsigned {
  kSiteBwdKvFull = 32, kSiteBwdEmpty, kSiteBwdFull, kSiteBwdDvDone, kSiteBwdDkDone, kSiteBwdPFull,
  kSiteBwdSFull, kSiteBwdAccDone, kSiteBwdDrain, kSiteBwdLoadDrain, kSiteBwdQFull, kSiteBwdDqDone,
  kSiteBwdDpFull, kSiteBwdDsFull
};

// A of the P.V-shaped MMAs (P^T, dS^T or dS) sits in TMEM as packed bf16:
// keys/queries 0-63 of the tile in columns [base, base + 32), 64-127 in
// [base + 64, base + 96) (each warpgroup packs over the start of its own half).
// K-step kk (16 values = 8 columns) therefore starts at this column.
__device__ __forceinline__ uint32_t bwd_packed_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// Byte offset of element (row r, k) in a 128 x 16 bf16 K-major operand without
// swizzle: 8 x 8 core matrices of 128 contiguous bytes, 128 bytes apart along
// K (LBO) and 256 bytes apart along the rows (SBO).
__host__ __device__ constexpr int bwd_seed_offset(int r, int k) {
  return (r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// v as the sum of three bf16 values (hi + mid + lo = v to about 2^-24 |v|),
// packed as the first three of eight bf16 in a 16-byte row chunk.
__device__ __forceinline__ uint4 bwd_seed_row(float v) {
  if (!(fabsf(v) < CUDART_INF_F)) {  // -inf (a row that sees no key): the first part carries it
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    return make_uint4(hi, 0u, 0u, 0u);
  }
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  return make_uint4(__bfloat16_as_ushort(hi) | (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16),
                    __bfloat16_as_ushort(lo), 0u, 0u);
}

// Per query row: lse2 = lse * log2(e) (+inf for a row that sees no key, so
// that its P is 0) and Dl = sum_t dO_t O_t in fp32 over the bf16 inputs.
// One 16-byte chunk per thread; the D/8 threads of a row reduce by shuffles.
template <int D>
__global__ void bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                const float* __restrict__ lse, float* __restrict__ lse2, float* __restrict__ dl,
                                uint8_t* __restrict__ seed_l, uint8_t* __restrict__ seed_d, float scale,
                                long long heads, int Nq, int Nq_pad) {
  constexpr int TPR = D / 8;
  const long long n = heads * Nq_pad * TPR;
  const long long stride = (long long)gridDim.x * blockDim.x;  // a multiple of 32
  const int lane = threadIdx.x & 31;
  for (long long base = (blockIdx.x * (long long)blockDim.x + threadIdx.x) - lane; base < n; base += stride) {
    const long long e = base + lane;
    const bool valid = e < n;
    const long long row = e / TPR;
    const int c = (int)(e % TPR);
    const int i = (int)(row % Nq_pad);
    const long long hh = row / Nq_pad;
    float acc = 0.f;
    if (valid && i < Nq) {
      const size_t off = ((size_t)hh * Nq + i) * D + 8 * c;
      const uint4 wo = *reinterpret_cast<const uint4*>(o + off);
      const uint4 wd = *reinterpret_cast<const uint4*>(dout + off);
      const uint32_t po[4] = {wo.x, wo.y, wo.z, wo.w}, pd[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc = fmaf(__uint_as_float(po[k] << 16), __uint_as_float(pd[k] << 16), acc);
        acc = fmaf(__uint_as_float(po[k] & 0xffff0000u), __uint_as_float(pd[k] & 0xffff0000u), acc);
      }
    }
#pragma unroll
    for (int m = TPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (valid && c == 0) {
      float l2 = CUDART_INF_F;
      if (i < Nq) {
        const float l = lse[(size_t)hh * Nq + i];
        l2 = l == -CUDART_INF_F ? CUDART_INF_F : l * 1.4426950408889634f;
      }
      const float d = i < Nq ? acc : 0.f;
      lse2[(size_t)hh * Nq_pad + i] = l2;
      dl[(size_t)hh * Nq_pad + i] = d;
      // Seeds of the dK/dV kernel: -lse/scale, so that (S^T + seed) scale
      // log2 e = S^T scale log2 e - lse2 (-inf for rows whose P is 0), and -Dl.
      const size_t tile = (size_t)hh * (Nq_pad / 128) + i / 128;
      const int r = i & 127;
      const float vl = l2 == CUDART_INF_F ? -CUDART_INF_F : -l2 / (scale * 1.4426950408889634f);
      *reinterpret_cast<uint4*>(seed_l + tile * 4096 + bwd_seed_offset(r, 0)) = bwd_seed_row(vl);
      *reinterpret_cast<uint4*>(seed_l + tile * 4096 + bwd_seed_offset(r, 8)) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(seed_d + tile * 4096 + bwd_seed_offset(r, 0)) = bwd_seed_row(-d);
      *reinterpret_cast<uint4*>(seed_d + tile * 4096 + bwd_seed_offset(r, 8)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Shared epilogue: 32 fp32 columns of the thread's TMEM lane, times `mul`,
// rounded to bf16 and stored to dst (or zeros when there is no accumulator).
__device__ __forceinline__ void bwd_store32(uint32_t taddr, bool have, float mul, __nv_bfloat16* dst, bool store) {
  uint32_t r[32];
  if (have) {
    tmem_ld32(taddr, r);
    tmem_wait_ld();
    tmem_reg_fence(r);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = 0u;
  }
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
  if (store) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  }
}

// ============================================================== dK, dV
template <int D>
__global__ void __launch_bounds__(352, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::KV_K_OFF;
  uint8_t* sV = smem + C::KV_V_OFF;
  uint8_t* sQ = smem + C::KV_Q_OFF;
  uint8_t* sDO = smem + C::KV_DO_OFF;
  uint8_t* sSEED = smem + C::KV_SEED_OFF;
  uint8_t* sONES = smem + C::KV_ONES_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::KV_BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + C::STAGES;
  uint64_t* s_full = empty + C::STAGES;  // S^T in TMEM
  uint64_t* dp_full = s_full + 1;        // dP^T in TMEM
  uint64_t* p_full = dp_full + 1;        // [2] warpgroup g wrote P^T of its half
  uint64_t* ds_full = p_full + 2;        // [2] warpgroup g wrote dS^T of its half
  uint64_t* dv_done = ds_full + 2;
  uint64_t* dk_done = dv_done + 1;
  uint64_t* acc_done = dk_done + 1;
  uint64_t* drain = acc_done + 1;
  uint64_t* stall_bar = drain + 1;  // test hook only: never arrived on
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::KV_MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::KV_MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Launch order: KV heads in pairs, and within a pair key tile 0 (the most
  // query tiles under causal masking) first, alternating between the two
  // heads. The CTAs running at once then share two heads' Q and dO in L2
  // instead of streaming every head's, and the heaviest tiles still go first.
  const int kt = blockIdx.x >> 1;
  const int hkv = 2 * blockIdx.y + (blockIdx.x & 1);
  if (hkv >= a.Hkv) return;  // odd head count: the last pair has one head (before any setup)
  const int b = blockIdx.z;
  const int key0 = kt * 128;
  // Query tiles holding a row that sees some key of this tile: [qt0, n_qt).
  const int n_qt = (a.Nq + 127) / 128;
  int qt0 = 0;
  if (a.causal) {
    const long long first = (long long)key0 - a.causal_offset;  // first query row that sees key0
    qt0 = first <= 0 ? 0 : (int)min((long long)n_qt, first / 128);
  }
  const int per_head = n_qt - qt0;
  const int n_steps = per_head * a.group;  // step n: head hkv*group + n / per_head, tile qt0 + n % per_head

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 2);  // released by both MMA issuers
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    for (int g = 0; g < 2; ++g) {
      mbar_init(p_full + g, 128);
      mbar_init(ds_full + g, 128);
    }
    mbar_init(dv_done, 1);
    mbar_init(dk_done, 1);
    mbar_init(acc_done, 1);
    mbar_init(drain, 2);  // one commit from each MMA issuer
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x < 256) {  // the seed MMAs' A operand: rows of (1, 1, 1, 0, ..., 0)
    const int r = threadIdx.x >> 1, khalf = threadIdx.x & 1;
    const uint32_t one = 0x3F80u;  // bf16 1.0
    *reinterpret_cast<uint4*>(sONES + bwd_seed_offset(r, 8 * khalf)) =
        khalf == 0 ? make_uint4(one | (one << 16), one, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // read by the tensor core (async proxy)
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_steps > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE_BYTES);
      const uint64_t stream_once = l2_policy_evict_first();  // this key tile is read by this CTA only
      for (int kb = 0; kb < C::KBLK; ++kb) {
        tma_load_3d_hint(sK + kb * C::BLOCK_BYTES, &tm_k, kv_full, kb * 64, key0, b * a.Hkv + hkv, stream_once);
        tma_load_3d_hint(sV + kb * C::BLOCK_BYTES, &tm_v, kv_full, kb * 64, key0, b * a.Hkv + hkv, stream_once);
      }
      int issued = 0;
      for (int n = 0; n < n_steps; ++n) {
        const int s = n % C::STAGES, u = n / C::STAGES;
        if (u > 0 && !mbar_wait(empty + s, (u - 1) & 1, a.status, kSiteBwdEmpty)) { *abort_flag = 1; break; }
        const int h = hkv * a.group + n / per_head;
        const int q0 = (qt0 + n % per_head) * 128;
        mbar_arrive_expect_tx(full + s, 2 * C::TILE_BYTES + 2 * C::SEED_BYTES);
        for (int kb = 0; kb < C::KBLK; ++kb) {
          tma_load_3d(sQ + s * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tm_q, full + s, kb * 64, q0, b * a.Hq + h);
          tma_load_3d(sDO + s * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tm_do, full + s, kb * 64, q0, b * a.Hq + h);
        }
        const size_t tile = (size_t)(b * a.Hq + h) * (a.Nq_pad / 128) + q0 / 128;
        bulk_load(sSEED + s * 2 * C::SEED_BYTES, a.seed_l + tile * C::SEED_BYTES, C::SEED_BYTES, full + s);
        bulk_load(sSEED + s * 2 * C::SEED_BYTES + C::SEED_BYTES, a.seed_d + tile * C::SEED_BYTES, C::SEED_BYTES,
                  full + s);
        issued = n + 1;
        if (*abort_flag) break;
      }
      if (*abort_flag) {
        // Let every copy still in flight land before the CTA exits.
        mbar_wait(kv_full, 0, a.status, kSiteBwdLoadDrain);
        for (int n = max(0, issued - C::STAGES); n < issued; ++n)
          mbar_wait(full + n % C::STAGES, (n / C::STAGES) & 1, a.status, kSiteBwdLoadDrain);
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // warp 9: S^T and dP^T; warp 10: dV and dK. The stage's Q and dO reach
    // warp 10's MMAs through warp 9's wait on the stage (whose S^T commit the
    // elementwise warps wait for before they release P^T).
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_ts = idesc_bf16_f32(128, D, true);
      constexpr uint32_t kHi = sw128_desc_hi(1024);
      constexpr uint32_t kTileW = C::TILE_BYTES >> 4;
      const uint32_t q_lo = sw128_desc_lo(smem_u32(sQ), 16), do_lo = sw128_desc_lo(smem_u32(sDO), 16);
      bool ok = true;
      if (warp == 9) {
        const uint32_t k_lo = sw128_desc_lo(smem_u32(sK), 16), v_lo = sw128_desc_lo(smem_u32(sV), 16);
        const uint64_t ones_desc = smem_desc_noswizzle(smem_u32(sONES), 128, 256);
        ok = mbar_wait(kv_full, 0, a.status, kSiteBwdKvFull, abort_flag);
        for (int n = 0; ok && n < n_steps; ++n) {
          const int s = n % C::STAGES;
          if (!(ok = mbar_wait(full + s, (n / C::STAGES) & 1, a.status, kSiteBwdFull, abort_flag))) break;
          const uint32_t seed_addr = smem_u32(sSEED + s * 2 * C::SEED_BYTES);
          // S^T = -lse/scale (seed MMA) + K Q^T; it overwrites P^T of the
          // previous step (read by its dV MMAs).
          if (n > 0 && !(ok = mbar_wait(dv_done, (n - 1) & 1, a.status, kSiteBwdDvDone, abort_flag))) break;
          tc_fence_after_sync();
          umma_ss(tmem + C::T_ST, ones_desc, smem_desc_noswizzle(seed_addr, 128, 256), idesc_ss, 0u);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = static_cast<uint32_t>(((kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32) >> 4);
            umma_ss_w(tmem + C::T_ST, k_lo + off, kHi, q_lo + s * kTileW + off, kHi, idesc_ss, 1u);
          }
          umma_commit(s_full);
          // dP^T = -Dl (seed MMA) + V dO^T; it overwrites dS^T of the previous
          // step (read by its dK MMAs).
          if (n > 0 && !(ok = mbar_wait(dk_done, (n - 1) & 1, a.status, kSiteBwdDkDone, abort_flag))) break;
          tc_fence_after_sync();
          umma_ss(tmem + C::T_DPT, ones_desc, smem_desc_noswizzle(seed_addr + C::SEED_BYTES, 128, 256), idesc_ss, 0u);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = static_cast<uint32_t>(((kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32) >> 4);
            umma_ss_w(tmem + C::T_DPT, v_lo + off, kHi, do_lo + s * kTileW + off, kHi, idesc_ss, 1u);
          }
          umma_commit(dp_full);
          umma_commit(empty + s);  // this issuer's reads of the stage
        }
      } else {
        // B operands (dO for dV, Q for dK) are MN-major here: K steps of 16 rows
        const uint32_t qm_lo = sw128_desc_lo(smem_u32(sQ), C::BLOCK_BYTES);
        const uint32_t dom_lo = sw128_desc_lo(smem_u32(sDO), C::BLOCK_BYTES);
        for (int n = 0; ok && n < n_steps; ++n) {
          const int s = n % C::STAGES;
          // dV += P^T dO, one half of the queries as soon as its warpgroup wrote P^T.
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (!(ok = mbar_wait(p_full + g, n & 1, a.status, kSiteBwdPFull, abort_flag))) break;
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 4 * g; kk < 4 * g + 4; ++kk)
              umma_ts_w(tmem + C::T_DV, tmem + C::T_ST + bwd_packed_col(kk), dom_lo + s * kTileW + kk * (16 * 128 >> 4),
                        kHi, idesc_ts, (n > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          umma_commit(dv_done);
          // dK += dS^T Q, likewise per half.
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (!(ok = mbar_wait(ds_full + g, n & 1, a.status, kSiteBwdDsFull, abort_flag))) break;
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 4 * g; kk < 4 * g + 4; ++kk)
              umma_ts_w(tmem + C::T_DK, tmem + C::T_DPT + bwd_packed_col(kk), qm_lo + s * kTileW + kk * (16 * 128 >> 4),
                        kHi, idesc_ts, (n > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          umma_commit(dk_done);
          umma_commit(empty + s);  // this issuer's reads of the stage
        }
        umma_commit(acc_done);
      }
      if (!ok) *abort_flag = 1;
      // Every MMA either issuer started has finished before TMEM is released
      // (the barrier completes once both have committed).
      umma_commit(drain);
      mbar_wait(drain, 0, a.status, kSiteBwdDrain);
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    const int g = warp >> 2;  // query columns [64g, 64g + 64) of every tile
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row in the tile
    const int kj = key0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tST = tmem + lane_off + C::T_ST + 64 * g, tDPT = tmem + lane_off + C::T_DPT + 64 * g;
    const float sl2 = a.scale_log2;
    bool ok = true;
    if (a.stall != 0 && g == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && n_steps > 0) {
      // test hook: in place of its first score wait, warpgroup 0 of block (0, 0, 0)
      // waits on a barrier nothing arrives on; it gives up after 1 ms and takes the
      // abort path. The backward's elementwise and copy waits do not watch the abort
      // flag (that keeps their polling light), so the other roles of the CTA give up
      // at their own limit; the status keeps the first site.
      mbar_wait(stall_bar, 0, a.status, kSiteBwdSFull, abort_flag, kStallLimitNs);
      ok = false;
    }
    for (int n = 0; ok && n < n_steps; ++n) {
      const int s = n % C::STAGES;
      const int q0 = (qt0 + n % per_head) * 128;
      if (!(ok = mbar_wait(s_full, n & 1, a.status, kSiteBwdSFull))) break;
      tc_fence_after_sync();
      // query q0 + 64g + c sees key kj iff c >= kj - causal_offset - q0 - 64g
      const bool need_mask = a.causal && key0 + 127 > q0 + 64 * g + a.causal_offset;
      const int cmin = kj - a.causal_offset - q0 - 64 * g;
      // ---- phase 1: P^T = exp2((S^T - lse/scale) scale log2 e), kept in fp32 for phase 2
      float p[64];
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        uint32_t sr[32];
        tmem_ld32(tST + 32 * pass, sr);
        tmem_wait_ld();
        tmem_reg_fence(sr);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 32 * pass + 2 * i;
          float x0, x1;
          fma2(x0, x1, __uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]), sl2, sl2, 0.f, 0.f);
          float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          if (need_mask) {
            p0 = c < cmin ? 0.f : p0;
            p1 = c + 1 < cmin ? 0.f : p1;
          }
          p[c] = p0;
          p[c + 1] = p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tST + 16 * pass, pk);  // over columns this warpgroup has already read
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(p_full + g);
      // ---- phase 2: dS^T = P^T (dP^T - Dl), the accumulator already holding dP^T - Dl
      if (!(ok = mbar_wait(dp_full, n & 1, a.status, kSiteBwdDpFull))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        uint32_t dr[32];
        tmem_ld32(tDPT + 32 * pass, dr);
        tmem_wait_ld();
        tmem_reg_fence(dr);
        uint32_t dk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 32 * pass + 2 * i;
          dk[i] = pack_bf16x2(p[c] * __uint_as_float(dr[2 * i]), p[c + 1] * __uint_as_float(dr[2 * i + 1]));
        }
        tmem_st16(tDPT + 16 * pass, dk);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(ds_full + g);
    }
    if (!ok) *abort_flag = 1;
    // ---------------------------------------------------------- epilogue
    bool have = false;
    if (ok && n_steps > 0) {
      have = ok = mbar_wait(acc_done, 0, a.status, kSiteBwdAccDone);
      tc_fence_after_sync();
      if (*abort_flag) have = false;
    }
    have = __all_sync(0xffffffffu, have);  // guards warp-collective TMEM loads
    // warpgroup 0 writes dV, warpgroup 1 writes dK (times the score scale)
    const bool in_range = kj < a.Nk;
    __nv_bfloat16* dst = (g == 0 ? a.dv : a.dk) + ((size_t)(b * a.Hkv + hkv) * a.Nk + (in_range ? kj : 0)) * D;
    const uint32_t col = g == 0 ? C::T_DV : C::T_DK;
    const float mul = g == 0 ? 1.f : a.scale;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) bwd_store32(tmem + lane_off + col + 32 * c, have, mul, dst + 32 * c, in_range);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ============================================================== dQ
template <int D>
__global__ void __launch_bounds__(352, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::Q_Q_OFF;
  uint8_t* sDO = smem + C::Q_DO_OFF;
  uint8_t* sK = smem + C::Q_K_OFF;
  uint8_t* sV = smem + C::Q_V_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::Q_BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + C::STAGES;
  uint64_t* s_full = empty + C::STAGES;
  uint64_t* s_free = s_full + 1;         // the elementwise warps read S into registers
  uint64_t* dp_full = s_free + 1;        // [2] per dP buffer
  uint64_t* ds_full = dp_full + 2;       // [2][2] dP buffer b, warpgroup g wrote dS of its half: 2b + g
  uint64_t* dq_done = ds_full + 4;       // [2] per dP buffer
  uint64_t* acc_done = dq_done + 2;
  uint64_t* drain = acc_done + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::Q_MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::Q_MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int n_qt = (a.Nq + 127) / 128;
  const int qt = n_qt - 1 - blockIdx.y;  // latest (most key tiles under causal masking) first
  const int b = blockIdx.z;
  const int hkv = h / a.group;
  const int q0 = qt * 128;
  // Key tiles [0, n_kt): up to the last key the tile's last row sees.
  const int last = min(q0 + 127, a.Nq - 1);
  const long long hi = a.causal ? min((long long)a.Nk - 1, (long long)last + a.causal_offset) : a.Nk - 1;
  const int n_kt = hi >= 0 ? (int)(hi / 128) + 1 : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 2);  // released by both MMA issuers
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(dp_full + i, 1);
      mbar_init(ds_full + 2 * i, 128);
      mbar_init(ds_full + 2 * i + 1, 128);
      mbar_init(dq_done + i, 1);
    }
    mbar_init(acc_done, 1);
    mbar_init(drain, 2);  // one commit from each MMA issuer
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
    if (lane == 0 && n_kt > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, 2 * C::TILE_BYTES);
      const uint64_t stream_once = l2_policy_evict_first();  // this query tile is read by this CTA only
      for (int kb = 0; kb < C::KBLK; ++kb) {
        tma_load_3d_hint(sQ + kb * C::BLOCK_BYTES, &tm_q, q_full, kb * 64, q0, b * a.Hq + h, stream_once);
        tma_load_3d_hint(sDO + kb * C::BLOCK_BYTES, &tm_do, q_full, kb * 64, q0, b * a.Hq + h, stream_once);
      }
      int issued = 0;
      for (int n = 0; n < n_kt; ++n) {
        const int s = n % C::STAGES, u = n / C::STAGES;
        if (u > 0 && !mbar_wait(empty + s, (u - 1) & 1, a.status, kSiteBwdEmpty)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(full + s, 2 * C::TILE_BYTES);
        for (int kb = 0; kb < C::KBLK; ++kb) {
          tma_load_3d(sK + s * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tm_k, full + s, kb * 64, n * 128,
                      b * a.Hkv + hkv);
          tma_load_3d(sV + s * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tm_v, full + s, kb * 64, n * 128,
                      b * a.Hkv + hkv);
        }
        issued = n + 1;
        if (*abort_flag) break;
      }
      if (*abort_flag) {
        mbar_wait(q_full, 0, a.status, kSiteBwdLoadDrain);
        for (int n = max(0, issued - C::STAGES); n < issued; ++n)
          mbar_wait(full + n % C::STAGES, (n / C::STAGES) & 1, a.status, kSiteBwdLoadDrain);
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // warp 9: S(n) and dP(n); warp 10: dQ. The stage's K reaches warp 10's
    // MMAs through warp 9's wait on the stage (whose S commit the elementwise
    // warps wait for before they release dS).
    if (lane == 0 && n_kt > 0) {
      constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_ts = idesc_bf16_f32(128, D, true);
      constexpr uint32_t kHi = sw128_desc_hi(1024);
      constexpr uint32_t kTileW = C::TILE_BYTES >> 4;
      bool ok = true;
      if (warp == 9) {
        const uint32_t q_lo = sw128_desc_lo(smem_u32(sQ), 16), do_lo = sw128_desc_lo(smem_u32(sDO), 16);
        const uint32_t k_lo = sw128_desc_lo(smem_u32(sK), 16), v_lo = sw128_desc_lo(smem_u32(sV), 16);
        ok = mbar_wait(q_full, 0, a.status, kSiteBwdQFull, abort_flag);
        // Every wait below is on a barrier that cannot run two phases ahead of
        // the one waited for (parity waits cannot tell those apart): S(n+1)
        // needs s_free(n), dP(n+2) needs dQ(n) through dq_done of its buffer.
        for (int n = 0; ok && n < n_kt; ++n) {
          const int s = n % C::STAGES;
          if (!(ok = mbar_wait(full + s, (n / C::STAGES) & 1, a.status, kSiteBwdFull, abort_flag))) break;
          // S(n) = Q K_n^T, once the elementwise warps have read S(n-1) into registers.
          if (n >= 1 && !(ok = mbar_wait(s_free, (n - 1) & 1, a.status, kSiteBwdSFull, abort_flag))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = static_cast<uint32_t>(((kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32) >> 4);
            umma_ss_w(tmem + C::T_S, q_lo + off, kHi, k_lo + s * kTileW + off, kHi, idesc_ss, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full);
          // dP(n) = dO V_n^T into dP buffer n & 1, which held dS(n-2) (read by dQ(n-2)).
          if (n >= 2 && !(ok = mbar_wait(dq_done + (n & 1), ((n >> 1) - 1) & 1, a.status, kSiteBwdDqDone, abort_flag)))
            break;
          tc_fence_after_sync();
          const uint32_t dst = tmem + ((n & 1) ? C::T_DP1 : C::T_DP0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = static_cast<uint32_t>(((kk >> 2) * C::BLOCK_BYTES + (kk & 3) * 32) >> 4);
            umma_ss_w(dst, do_lo + off, kHi, v_lo + s * kTileW + off, kHi, idesc_ss, kk > 0 ? 1u : 0u);
          }
          umma_commit(dp_full + (n & 1));
          umma_commit(empty + s);  // this issuer's reads of the stage
        }
      } else {
        const uint32_t km_lo = sw128_desc_lo(smem_u32(sK), C::BLOCK_BYTES);  // MN-major K: steps of 16 keys
        for (int n = 0; ok && n < n_kt; ++n) {
          const int s = n % C::STAGES;
          // dQ += dS K, one half of the keys as soon as its warpgroup wrote dS
          // (dS(n) sits in dP buffer n & 1).
          const uint32_t dp = tmem + ((n & 1) ? C::T_DP1 : C::T_DP0);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (!(ok = mbar_wait(ds_full + 2 * (n & 1) + g, (n >> 1) & 1, a.status, kSiteBwdDsFull, abort_flag))) break;
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 4 * g; kk < 4 * g + 4; ++kk)
              umma_ts_w(tmem + C::T_DQ, dp + bwd_packed_col(kk), km_lo + s * kTileW + kk * (16 * 128 >> 4), kHi,
                        idesc_ts, (n > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          umma_commit(dq_done + (n & 1));
          umma_commit(empty + s);  // this issuer's reads of the stage
        }
        umma_commit(acc_done);
      }
      if (!ok) *abort_flag = 1;
      // Every MMA either issuer started has finished before TMEM is released
      // (the barrier completes once both have committed).
      umma_commit(drain);
      mbar_wait(drain, 0, a.status, kSiteBwdDrain);
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    const int g = warp >> 2;  // key columns [64g, 64g + 64) of every tile
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int qi = q0 + r;  // < Nq_pad
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;

    const float sl2 = a.scale_log2;
    const float lse2 = a.lse2[(size_t)(b * a.Hq + h) * a.Nq_pad + qi];
    const float dl = a.dl[(size_t)(b * a.Hq + h) * a.Nq_pad + qi];
    // last key this row sees (keys past it are masked)
    const long long lim_ll = a.causal ? min((long long)a.Nk - 1, (long long)qi + a.causal_offset) : a.Nk - 1;
    const int lim = (int)max(lim_ll, -1LL);
    // the tile needs masking when a row's limit falls inside it (tile-uniform test on the first row)
    const long long lim_first = a.causal ? min((long long)a.Nk - 1, (long long)q0 + a.causal_offset) : a.Nk - 1;
    bool ok = true;
    for (int n = 0; ok && n < n_kt; ++n) {
      if (!(ok = mbar_wait(s_full, n & 1, a.status, kSiteBwdSFull))) break;
      tc_fence_after_sync();
      const uint32_t tS = tmem + lane_off + C::T_S + 64 * g;
      const uint32_t tDP = tmem + lane_off + ((n & 1) ? C::T_DP1 : C::T_DP0) + 64 * g;
      const int kbase = n * 128 + 64 * g;
      const bool need_mask = kbase + 63 > lim_first;
      const int cmax = lim - kbase;  // column c is visible iff c <= cmax
      // ---- phase 1: P = exp2(S scale log2 e - lse2)
      float p[64];
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        uint32_t sr[32];
        tmem_ld32(tS + 32 * pass, sr);
        tmem_wait_ld();
        tmem_reg_fence(sr);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 32 * pass + 2 * i;
          float x0, x1;
          fma2(x0, x1, __uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]), sl2, sl2, -lse2, -lse2);
          float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          if (need_mask) {
            p0 = c > cmax ? 0.f : p0;
            p1 = c + 1 > cmax ? 0.f : p1;
          }
          p[c] = p0;
          p[c + 1] = p1;
        }
      }
      // S(n) is in registers: the S issuer may compute S(n+1) into its columns
      tc_fence_before_sync();
      mbar_arrive(s_free);
      // ---- phase 2: dS = P (dP - Dl), packed over this half's first 32 columns of dP
      if (!(ok = mbar_wait(dp_full + (n & 1), (n >> 1) & 1, a.status, kSiteBwdDpFull))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        uint32_t dr[32];
        tmem_ld32(tDP + 32 * pass, dr);
        tmem_wait_ld();
        tmem_reg_fence(dr);
        uint32_t dk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 32 * pass + 2 * i;
          float d0, d1;
          fma2(d0, d1, __uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]), 1.f, 1.f, -dl, -dl);
          dk[i] = pack_bf16x2(p[c] * d0, p[c + 1] * d1);
        }
        tmem_st16(tDP + 16 * pass, dk);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(ds_full + 2 * (n & 1) + g);
    }
    if (!ok) *abort_flag = 1;
    // ---------------------------------------------------------- epilogue
    bool have = false;
    if (ok && n_kt > 0) {
      have = ok = mbar_wait(acc_done, 0, a.status, kSiteBwdAccDone);
      tc_fence_after_sync();
      if (*abort_flag) have = false;
    }
    have = __all_sync(0xffffffffu, have);  // guards warp-collective TMEM loads
    const bool in_range = qi < a.Nq;
    __nv_bfloat16* dst = a.dq + ((size_t)(b * a.Hq + h) * a.Nq + (in_range ? qi : 0)) * D;
    // warpgroup g writes columns [g D/2, (g+1) D/2)
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      const int col = g * (D / 2) + 32 * c;
      bwd_store32(tmem + lane_off + C::T_DQ + col, have, a.scale, dst + col, in_range);
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
