// KV-cache decode for sm_103a: one new query token per sequence attends to
// the cached keys/values 0..seqlens[b]-1 ([IMR] prefill/decode section;
// [PW] §3.1-§3.2), with MHA/GQA/MQA head sharing ([PW] §2.3).
//
// Sources: [IMR] imreese.github.io "Transformer 笔记：注意力机制为什么会变成系统问题";
// [PW] pwwt.cn news 6124947; [MG-A] menggq.pages.dev "Transformer 架构的数学与
// 计算深度解析" (§6.3, two-block merge); [AUT] auturnal.com "从注意力到 IO 感知执行" (§8).
//
// The work is bound by reading the cache, so it runs on the CUDA cores: the
// contraction per key is only GC x D multiply-adds for 2*D*2 bytes read.
// Grid: (split, (b, kv head, query group)). Each CTA streams its split of the
// cache through a ring of TMA-loaded 64-key tiles (128-byte swizzled, so the
// per-key row reads below are bank-conflict free), keeps the blockwise softmax
// statistics (m, l, un-normalised u) of [AUT] §8 for each of its GC query
// heads, and writes a partial (o = u / l, lse). The last CTA of a
// (b, kv head, query group) to finish merges the partials with the two-block
// rule of [MG-A] §6.3 generalised to n blocks, and resets its ticket.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "ptx.cuh"

namespace attn_dev {

struct DecArgs {
  const __nv_bfloat16* q;  // [B, Hq, D]
  const int* seqlens;      // [B]
  __nv_bfloat16* o;        // [B, Hq, D]
  float* lse;              // [B, Hq] natural-log LSE, or nullptr
  float* part_o;           // [units][max_splits][GC][D]   (workspace)
  float* part_lse;         // [units][max_splits][GC]      (workspace, base-2 units)
  int* tickets;            // [units]                      (workspace, zero between calls)
  int B, Hq, Hkv, Lmax;
  int group;               // Hq / Hkv
  int qgroups;             // group / GC
  int split;               // keys per split (multiple of 64)
  int max_splits;          // ceil(Lmax / split)
  float scale_log2;        // scale * log2(e)
  unsigned* status;
};

template <int D, int GC>
struct DecCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(GC == 1 || GC == 2 || GC == 4 || GC == 8, "query heads per CTA");
  static constexpr int THREADS = 256;
  static constexpr int TK = 64;                      // keys per tile
  static constexpr int KBLK = D / 64;                // 128-byte swizzle blocks per row
  static constexpr int BOX_BYTES = TK * 64 * 2;      // 64 keys x 64 columns
  static constexpr int TILE_BYTES = KBLK * BOX_BYTES;  // K (or V) tile
  static constexpr int STAGES = 3;
  static constexpr int KV_OFF = 0;                   // stage s: K at 2s, V at 2s+1
  static constexpr int Q_OFF = KV_OFF + STAGES * 2 * TILE_BYTES;
  static constexpr int S_OFF = Q_OFF + GC * D * 4;   // scores [GC][TK]
  static constexpr int P_OFF = S_OFF + GC * TK * 4;  // probabilities [TK][GC]
  static constexpr int A_OFF = P_OFF + GC * TK * 4;  // alpha [GC], m [GC], l [GC]
  static constexpr int BAR_OFF = A_OFF + 3 * 8 * 4;
  static constexpr int MISC_OFF = BAR_OFF + STAGES * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
  // cross-warp reduction of the value accumulators reuses the K/V ring
  static_assert(8 * GC * D * 4 <= STAGES * 2 * TILE_BYTES, "reduction scratch");
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D, int GC>
__global__ void __launch_bounds__(256)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const DecArgs a) {
  using C = DecCfg<D, GC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* q_s = reinterpret_cast<float*>(smem + C::Q_OFF);   // [GC][D], pre-scaled by scale*log2(e)
  float* s_s = reinterpret_cast<float*>(smem + C::S_OFF);   // [GC][TK]
  float* p_s = reinterpret_cast<float*>(smem + C::P_OFF);   // [TK][GC]
  float* alpha_s = reinterpret_cast<float*>(smem + C::A_OFF);
  float* m_s = alpha_s + 8;
  float* l_s = alpha_s + 16;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  int* flag_s = reinterpret_cast<int*>(smem + C::MISC_OFF);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int split_idx = blockIdx.x;
  const int unit = blockIdx.y;                  // (b, hkv, qg)
  const int qg = unit % a.qgroups;
  const int bh = unit / a.qgroups;
  const int hkv = bh % a.Hkv;
  const int b = bh / a.Hkv;
  const int h0 = hkv * a.group + qg * GC;       // first query head of this CTA

  int L = a.seqlens[b];
  if (L < 0 || L > a.Lmax) {
    if (split_idx == 0 && tid == 0) atomicOr(a.status, kStatusBadSeqlen);
    L = max(0, min(L, a.Lmax));
  }
  const int n_splits = (L + a.split - 1) / a.split;
  if (L == 0) {
    // No cached key: o = 0, lse = -inf.
    if (split_idx == 0) {
      for (int i = tid; i < GC * D; i += C::THREADS)
        a.o[(size_t)(b * a.Hq + h0 + i / D) * D + i % D] = __float2bfloat16_rn(0.f);
      if (a.lse != nullptr && tid < GC) a.lse[b * a.Hq + h0 + tid] = -CUDART_INF_F;
    }
    return;
  }
  if (split_idx >= n_splits) return;
  const int k_begin = split_idx * a.split;
  const int k_end = min(L, k_begin + a.split);
  const int n_tiles = (k_end - k_begin + C::TK - 1) / C::TK;

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) mbar_init(full + s, 1);
    *flag_s = 0;
    fence_mbarrier_init();
  }
  for (int i = tid; i < GC * D; i += C::THREADS) {
    const float qv = __bfloat162float(a.q[(size_t)(b * a.Hq + h0 + i / D) * D + i % D]);
    q_s[i] = qv * a.scale_log2;
  }
  __syncthreads();

  auto issue = [&](int tile) {
    const int s = tile % C::STAGES;
    uint8_t* kdst = smem + C::KV_OFF + (2 * s) * C::TILE_BYTES;
    uint8_t* vdst = kdst + C::TILE_BYTES;
    mbar_arrive_expect_tx(full + s, 2 * C::TILE_BYTES);
    const int key = k_begin + tile * C::TK;
#pragma unroll
    for (int kb = 0; kb < C::KBLK; ++kb) {
      tma_load_3d(kdst + kb * C::BOX_BYTES, &tm_k, full + s, kb * 64, key, b * a.Hkv + hkv);
      tma_load_3d(vdst + kb * C::BOX_BYTES, &tm_v, full + s, kb * 64, key, b * a.Hkv + hkv);
    }
  };
  int issued = 0;  // tiles whose loads thread 0 has issued
  if (tid == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int t = 0; t < C::STAGES - 1 && t < n_tiles; ++t) issue(t), ++issued;
  }

  // QK mapping: thread -> (key within tile, query subset)
  const int qk_key = tid & (C::TK - 1);
  const int qk_sel = tid >> 6;                       // 0..3, warp-uniform
  constexpr int QPT = GC >= 4 ? GC / 4 : 1;          // queries per thread
  const bool qk_active = GC >= 4 || qk_sel < GC;
  // PV mapping: warp -> keys w, w+8, ...; lane -> EPL consecutive value columns
  constexpr int EPL = D / 32;
  float acc[GC][EPL];
#pragma unroll
  for (int g = 0; g < GC; ++g)
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
  float m_run = -CUDART_INF_F, l_run = 0.f;  // owned by warp g (< GC), replicated over its lanes
  bool ok = true;

  for (int tile = 0; tile < n_tiles; ++tile) {
    const int s = tile % C::STAGES;
    const uint8_t* ks = smem + C::KV_OFF + (2 * s) * C::TILE_BYTES;
    const uint8_t* vs = ks + C::TILE_BYTES;
    if (!mbar_wait(full + s, (tile / C::STAGES) & 1, a.status, 20)) ok = false;
    if (!ok) *flag_s = 1;
    const int key0 = k_begin + tile * C::TK;
    // ---- scores: s[g][key] = (scale*log2e) q_g . k_key
    if (qk_active) {
      float dot[QPT];
#pragma unroll
      for (int i = 0; i < QPT; ++i) dot[i] = 0.f;
      const int sw = qk_key & 7;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint8_t* rowp = ks + (c >> 3) * C::BOX_BYTES + qk_key * 128;
        const uint4 kw = *reinterpret_cast<const uint4*>(rowp + (((c & 7) ^ sw) << 4));
        float kf[8] = {bf16lo(kw.x), bf16hi(kw.x), bf16lo(kw.y), bf16hi(kw.y),
                       bf16lo(kw.z), bf16hi(kw.z), bf16lo(kw.w), bf16hi(kw.w)};
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
          const int g = qk_sel + 4 * i;
          const float4 qa = *reinterpret_cast<const float4*>(q_s + g * D + 8 * c);
          const float4 qb = *reinterpret_cast<const float4*>(q_s + g * D + 8 * c + 4);
          dot[i] = fmaf(qa.x, kf[0], dot[i]);
          dot[i] = fmaf(qa.y, kf[1], dot[i]);
          dot[i] = fmaf(qa.z, kf[2], dot[i]);
          dot[i] = fmaf(qa.w, kf[3], dot[i]);
          dot[i] = fmaf(qb.x, kf[4], dot[i]);
          dot[i] = fmaf(qb.y, kf[5], dot[i]);
          dot[i] = fmaf(qb.z, kf[6], dot[i]);
          dot[i] = fmaf(qb.w, kf[7], dot[i]);
        }
      }
      const bool valid = key0 + qk_key < k_end;
#pragma unroll
      for (int i = 0; i < QPT; ++i) s_s[(qk_sel + 4 * i) * C::TK + qk_key] = valid ? dot[i] : -CUDART_INF_F;
    }
    __syncthreads();
    // Flags are only written before the barrier above, so every thread takes
    // the same branch here.
    if (*flag_s) break;
    // The stage read two tiles ago is free now: refill it.
    if (tid == 0 && tile + C::STAGES - 1 < n_tiles) issue(tile + C::STAGES - 1), ++issued;
    // ---- online softmax update, one warp per query head
    if (warp < GC) {
      const float s0 = s_s[warp * C::TK + lane];
      const float s1 = s_s[warp * C::TK + lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_run, mx);       // finite: every tile has a valid key
      const float alpha = ex2_approx(m_run - m_new);
      const float p0 = ex2_approx(s0 - m_new);
      const float p1 = ex2_approx(s1 - m_new);
      float sum = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      p_s[lane * GC + warp] = p0;
      p_s[(lane + 32) * GC + warp] = p1;
      if (lane == 0) alpha_s[warp] = alpha;
    }
    __syncthreads();
    // ---- u = alpha u + sum_k p_k v_k
#pragma unroll
    for (int g = 0; g < GC; ++g) {
      const float al = alpha_s[g];
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[g][e] *= al;
    }
    const int e0 = lane * EPL;              // first value column of this lane
    const int vblk = e0 >> 6;               // 64-column swizzle block
    const int vchunk = (e0 & 63) >> 3;      // 16-byte chunk inside the 128-byte row
    const int vin = (e0 & 7) * 2;           // byte offset inside the chunk
    const int n_valid = min(C::TK, k_end - key0);  // rows past the length are never touched
#pragma unroll 2
    for (int kk = warp; kk < n_valid; kk += 8) {
      const uint8_t* rowp = vs + vblk * C::BOX_BYTES + kk * 128 + (((vchunk ^ (kk & 7)) << 4) + vin);
      float vf[EPL];
      if constexpr (EPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(rowp);
        vf[0] = bf16lo(w.x); vf[1] = bf16hi(w.x); vf[2] = bf16lo(w.y); vf[3] = bf16hi(w.y);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(rowp);
        vf[0] = bf16lo(w); vf[1] = bf16hi(w);
      }
      float pg[GC];
      if constexpr (GC >= 4) {
#pragma unroll
        for (int g4 = 0; g4 < GC; g4 += 4) {
          const float4 pp = *reinterpret_cast<const float4*>(p_s + kk * GC + g4);
          pg[g4] = pp.x; pg[g4 + 1] = pp.y; pg[g4 + 2] = pp.z; pg[g4 + 3] = pp.w;
        }
      } else {
#pragma unroll
        for (int g = 0; g < GC; ++g) pg[g] = p_s[kk * GC + g];
      }
#pragma unroll
      for (int g = 0; g < GC; ++g)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(pg[g], vf[e], acc[g][e]);
    }
  }
  __syncthreads();
  if (*flag_s) {
    // A wait gave up: let the copies still in flight land, then leave.
    if (tid == 0)
      for (int t = max(0, issued - C::STAGES); t < issued; ++t)
        mbar_wait(full + t % C::STAGES, (t / C::STAGES) & 1, a.status, 21);
    return;
  }
  // Every issued tile was waited on above, so all loads have landed and the
  // ring is free for the cross-warp reduction.
  float* red = reinterpret_cast<float*>(smem + C::KV_OFF);  // [8][GC][D]
#pragma unroll
  for (int g = 0; g < GC; ++g)
#pragma unroll
    for (int e = 0; e < EPL; ++e) red[(warp * GC + g) * D + lane * EPL + e] = acc[g][e];
  if (warp < GC && lane == 0) {
    m_s[warp] = m_run;
    l_s[warp] = l_run;
  }
  __syncthreads();

  const size_t pbase = (size_t)unit * a.max_splits;
  if (n_splits == 1) {
    for (int i = tid; i < GC * D; i += C::THREADS) {
      const int g = i / D;
      float u = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) u += red[(w * GC + g) * D + i % D];
      a.o[(size_t)(b * a.Hq + h0 + g) * D + i % D] = __float2bfloat16_rn(u / l_s[g]);
    }
    if (a.lse != nullptr && tid < GC)
      a.lse[b * a.Hq + h0 + tid] = (m_s[tid] + log2f(l_s[tid])) * 0.69314718055994531f;
    return;
  }
  // Partial of this split: normalised o and its base-2 lse.
  for (int i = tid; i < GC * D; i += C::THREADS) {
    const int g = i / D;
    float u = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) u += red[(w * GC + g) * D + i % D];
    a.part_o[((pbase + split_idx) * GC + g) * D + i % D] = u / l_s[g];
  }
  if (tid < GC) a.part_lse[(pbase + split_idx) * GC + tid] = m_s[tid] + log2f(l_s[tid]);
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int ticket = atomicAdd(a.tickets + unit, 1);
    *flag_s = (ticket == n_splits - 1) ? 2 : 0;
  }
  __syncthreads();
  if (*flag_s != 2) return;
  // Last split to finish: merge all partials of this unit.
  __threadfence();
  if (tid < GC) {
    float mx = -CUDART_INF_F;
    for (int sp = 0; sp < n_splits; ++sp)
      mx = fmaxf(mx, __ldcg(a.part_lse + (pbase + sp) * GC + tid));
    float tot = 0.f;
    for (int sp = 0; sp < n_splits; ++sp) {
      const float w = ex2_approx(__ldcg(a.part_lse + (pbase + sp) * GC + tid) - mx);
      tot += w;
    }
    m_s[tid] = mx;
    l_s[tid] = tot;
    if (a.lse != nullptr) a.lse[b * a.Hq + h0 + tid] = (mx + log2f(tot)) * 0.69314718055994531f;
  }
  __syncthreads();
  for (int i = tid; i < GC * D; i += C::THREADS) {
    const int g = i / D;
    float u = 0.f;
    for (int sp = 0; sp < n_splits; ++sp) {
      const float w = ex2_approx(__ldcg(a.part_lse + (pbase + sp) * GC + g) - m_s[g]);
      u = fmaf(w, __ldcg(a.part_o + ((pbase + sp) * GC + g) * D + i % D), u);
    }
    a.o[(size_t)(b * a.Hq + h0 + g) * D + i % D] = __float2bfloat16_rn(u / l_s[g]);
  }
  if (tid == 0) a.tickets[unit] = 0;  // ready for the next call
}

}  // namespace attn_dev
