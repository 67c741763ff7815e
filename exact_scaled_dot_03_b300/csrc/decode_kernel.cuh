// KV-cache decode for sm_103a: one new query token per sequence attends to
// the cached keys/values 0..seqlens[b]-1 ([IMR] prefill/decode section;
// [PW] §3.1-§3.2), with MHA/GQA/MQA head sharing ([PW] §2.3).
//
// Sources: [IMR] imreese.github.io "Transformer 笔记：注意力机制为什么会变成系统问题";
// [PW] pwwt.cn news 6124947; [MG-A] menggq.pages.dev "Transformer 架构的数学与
// 计算深度解析" (§6.3, two-block merge); [AUT] auturnal.com "从注意力到 IO 感知执行" (§8).
//
// The work is bound by reading the cache. Its two contractions per KV head
// are small dense products (GC query heads x 16 keys x D per warp and tile);
// on the CUDA cores their issue cost (unpacking bf16, cross-lane sums) kept
// the kernel from saturating HBM, so they run as warp-level tensor-core MMAs
// (m16n8k16, bf16 in, fp32 accumulate) on fragments read with ldmatrix from
// the TMA-staged tiles; the kernel stays bound by the cache read.
//
// Work split (persistent, balanced). A "unit" is one (sequence b, KV head,
// group of GC query heads); its cache rows are cut into 128-key tiles. All
// units' tiles are laid end to end (sequence-major) and the grid (one CTA per
// SM) takes equal contiguous chunks of that list, so every CTA streams the
// same number of bytes whatever the length mix. A chunk covers the tail of
// one unit, whole units, and the head of another; each such "piece" ends in a
// result (o = u / l and its log-sum-exp). A unit covered by one piece is
// written out directly. Otherwise the piece is a partial result (at most two
// per CTA: its first and its last piece); once a CTA has streamed all its
// tiles it takes a ticket for each, and the last piece of a unit to finish
// merges the partials with the two-block rule of [MG-A] §6.3 generalised to
// n blocks, and resets the ticket.
//
// Inside a CTA: K and V tiles stream through a ring of STAGES TMA-loaded
// shared-memory stages (128-byte swizzle). Warp w owns keys [16 w, 16 w + 16)
// of every tile and keeps its own blockwise-softmax state ([AUT] §8: running
// max m, denominator l, un-normalised u) for the GC query heads, so no
// CTA-wide barrier is needed per tile; the last warp to finish with a stage
// refills it (a per-stage release counter, no producer warp). At the end of a
// piece every warp leaves its (m, l, u) in shared memory and, after one
// barrier, each thread merges two output elements over the warps (max,
// rescale, sum); the next piece's query fragments are loaded meanwhile.
//
// Per warp and tile: S = Q K^T as 2 x D/16 MMAs (query rows 0..GC-1 of the
// 16-row A operand; the rest are zero), the scale applied in fp32, the
// running max moved lazily (only when a tile's max exceeds it by more than 8
// in base-2 units; l and u always share it, so o = u / l is unchanged), P
// rounded to bf16 and fed back as the A operand of O += P V (D/8 MMAs).
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
  float* part_o;           // [units][slots][GC][D]   (workspace) normalised partial outputs
  float* part_lse;         // [units][slots][GC]      (workspace) partial LSE, base-2 units
  int* tickets;            // [units]                 (workspace, zero between calls)
  int B, Hq, Hkv, Lmax;
  int group;               // Hq / Hkv
  int qgroups;             // group / GC
  int slots;               // partial slots per unit (>= pieces any unit can be cut into)
  float scale_log2;        // scale * log2(e)
  unsigned* status;
  // Paged cache (block_table != nullptr): position p of sequence b is row
  // p % page_size of page block_table[b * bt_stride + p / page_size] of the
  // [num_pages, Hkv, page_size, D] cache; page_size divides 128 or is a
  // multiple of it. Otherwise the cache is [B, Hkv, Lmax, D].
  const int* block_table;
  int bt_stride, page_size, num_pages;
  // Fused append (k_new != nullptr): the new token's K/V [B, Hkv, D] is written
  // at position seqlens[b] of the cache and attended to with the cached keys.
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  // Failure-detection test hook: when set, warp 0 of block 0 replaces its first
  // tile wait by a wait on a barrier that nothing arrives on, with a 1 ms limit
  // (0 in normal use).
  int stall;
};

template <int D, int GC>
struct DecCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(GC == 1 || GC == 2 || GC == 4 || GC == 8, "query heads per unit");
  static constexpr int NW = 8;                   // warps; every warp consumes, any warp may refill
  static constexpr int THREADS = NW * 32;
  static constexpr int TK = 128;                 // keys per tile
  static constexpr int KPW = TK / NW;            // keys per warp per tile (one 16-key MMA step)
  static_assert(KPW == 16, "one k-step of the P.V MMA per warp");
  static constexpr int KBLK = D / 64;            // 64-column (128-byte) swizzle boxes per row
  static constexpr int BOX_BYTES = TK * 128;
  static constexpr int TILE_BYTES = KBLK * BOX_BYTES;  // K (or V) tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K then V
  static constexpr int STAGES = (D == 128) ? 3 : 6;
  static constexpr int MIN_CHUNK = 4;            // tiles: bounds the pieces a unit is cut into
  // shared memory
  static constexpr int RING_OFF = 0;
  static constexpr int SL_OFF = RING_OFF + STAGES * STAGE_BYTES;  // [NW][GC][D] per-warp u
  static constexpr int WM_OFF = SL_OFF + NW * GC * D * 4;         // [NW][GC] per-warp running max
  static constexpr int WL_OFF = WM_OFF + NW * GC * 4;             // [NW][GC] per-warp denominator
  static constexpr int BAR_OFF = WL_OFF + NW * GC * 4;            // full[STAGES]
  static constexpr int CNT_OFF = BAR_OFF + STAGES * 8;            // releases[STAGES], fills[STAGES]
  // abort flag, last flags, plan (3 x int64 at +16), the test hook's barrier at +48
  static constexpr int MISC_OFF = CNT_OFF + 2 * STAGES * 4 + 8;
  static_assert(MISC_OFF % 8 == 0, "mbarrier and int64 alignment");
  static constexpr int SMEM_BYTES = MISC_OFF + 64 + 1024;         // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// Position in the CTA's tile list: sequence b (nt tiles per unit, list offset
// P of its first unit), unit r within the sequence, tile j within the unit.
struct TileCursor {
  int b, nt, r, j;
  long long P;
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Keys sequence b attends to: its cached length, clamped into
// [0, Lmax - 1 if appending else Lmax], plus the appended token.
__device__ __forceinline__ int dec_len(const DecArgs& a, int b) {
  const int app = a.k_new != nullptr ? 1 : 0;
  const int L = a.seqlens[b];
  return max(0, min(L, a.Lmax - app)) + app;
}

// Physical page holding logical page lp of sequence b (flagged and replaced
// by page 0 when the table holds an id outside [0, num_pages)).
__device__ __forceinline__ int dec_page(const DecArgs& a, int b, int lp) {
  const int pg = a.block_table[(size_t)b * a.bt_stride + lp];
  if (pg < 0 || pg >= a.num_pages) {
    atomicOr(a.status, kStatusBadPage);
    return 0;
  }
  return pg;
}

// Element offset of the cache row holding position p of (sequence b, KV head hkv).
__device__ __forceinline__ size_t dec_row_offset(const DecArgs& a, int b, int hkv, int p, int D) {
  if (a.block_table == nullptr) return (((size_t)b * a.Hkv + hkv) * a.Lmax + p) * D;
  const int pg = dec_page(a, b, p / a.page_size);
  return (((size_t)pg * a.Hkv + hkv) * a.page_size + p % a.page_size) * D;
}

// Sum of x over the warp (all lanes receive it).
__device__ __forceinline__ long long warp_sum_ll(long long x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Wait sites recorded in status[1] when a bounded wait gives up.
enum : unsigned { kSiteDecFull = 20, kSiteDecDrain = 22 };

template <int TK>
__device__ __forceinline__ int dec_tiles(const DecArgs& a, int b) {
  return (dec_len(a, b) + TK - 1) / TK;
}

// Steps a cursor to the next tile in list order. Only called while a later
// tile exists, so the loop over empty sequences stops inside [0, B).
template <int TK>
__device__ __forceinline__ void dec_advance(const DecArgs& a, int UPB, TileCursor& c) {
  if (++c.j < c.nt) return;
  c.j = 0;
  if (++c.r < UPB) return;
  c.r = 0;
  c.P += (long long)c.nt * UPB;
  do {
    ++c.b;
    c.nt = dec_tiles<TK>(a, c.b);
  } while (c.nt == 0);
}

template <int D, int GC>
__global__ void __launch_bounds__(DecCfg<D, GC>::THREADS, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_k16, const __grid_constant__ CUtensorMap tm_v16,
                       const DecArgs a) {
  using C = DecCfg<D, GC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + C::RING_OFF;
  float* sl_sm = reinterpret_cast<float*>(smem + C::SL_OFF);
  float* wm_sm = reinterpret_cast<float*>(smem + C::WM_OFF);
  float* wl_sm = reinterpret_cast<float*>(smem + C::WL_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  int* releases = reinterpret_cast<int*>(smem + C::CNT_OFF);  // warps done with each stage (monotonic)
  int* fills = releases + C::STAGES;                          // loads issued into each stage
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF);
  volatile int* last_flag = abort_flag + 1;
  long long* plan_sm = reinterpret_cast<long long*>(smem + C::MISC_OFF + 16);  // T, b_start, P_start
  uint64_t* stall_bar = reinterpret_cast<uint64_t*>(smem + C::MISC_OFF + 48);  // test hook: never arrived on

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int UPB = a.Hkv * a.qgroups;  // units per sequence

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full + s, 1);
      releases[s] = 0;
      fills[s] = 0;
    }
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbarrier_init();
  }

  // ---- the tile list: total T, and the sequence this CTA's chunk starts in
  if (warp == 0) {
    bool bad = false;
    long long total = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      const int b = b0 + lane;
      long long tiles = 0;
      if (b < a.B) {
        const int L = a.seqlens[b];
        bad |= (L < 0 || L > a.Lmax - (a.k_new != nullptr ? 1 : 0));
        tiles = (long long)dec_tiles<C::TK>(a, b) * UPB;  // the same length rule as every walker below
      }
      total += warp_sum_ll(tiles);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (bad && blockIdx.x == 0 && lane == 0) atomicOr(a.status, kStatusBadSeqlen);
    const long long chunk = max((total + gridDim.x - 1) / gridDim.x, (long long)C::MIN_CHUNK);
    const long long t0 = (long long)blockIdx.x * chunk;
    if (lane == 0) {
      plan_sm[0] = total;
      plan_sm[1] = -1;
      plan_sm[2] = 0;
    }
    __syncwarp();
    if (t0 < total) {
      long long run = 0;
      for (int b0 = 0; b0 < a.B && run <= t0; b0 += 32) {
        const int b = b0 + lane;
        const long long tiles = b < a.B ? (long long)dec_tiles<C::TK>(a, b) * UPB : 0;
        long long incl = tiles;  // inclusive warp scan
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const long long y = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += y;
        }
        const long long lo = run + incl - tiles;
        if (tiles > 0 && t0 >= lo && t0 < lo + tiles) {
          plan_sm[1] = b;
          plan_sm[2] = lo;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  __syncthreads();

  // Sequences with no cached key: o = 0, lse = -inf.
  for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
    if (dec_len(a, b) != 0) continue;
    for (int i = tid; i < a.Hq * D; i += C::THREADS)
      a.o[(size_t)b * a.Hq * D + i] = __float2bfloat16_rn(0.f);
    if (a.lse != nullptr)
      for (int i = tid; i < a.Hq; i += C::THREADS) a.lse[(size_t)b * a.Hq + i] = -CUDART_INF_F;
  }

  const long long T = plan_sm[0];
  const long long chunk = max((T + gridDim.x - 1) / gridDim.x, (long long)C::MIN_CHUNK);
  const long long t0 = (long long)blockIdx.x * chunk;
  if (t0 >= T) return;  // uniform over the CTA
  const long long t1 = min(T, t0 + chunk);
  const int n_tiles = static_cast<int>(t1 - t0);

  TileCursor cur;
  cur.b = static_cast<int>(plan_sm[1]);
  cur.P = plan_sm[2];
  cur.nt = dec_tiles<C::TK>(a, cur.b);
  cur.r = static_cast<int>((t0 - cur.P) / cur.nt);
  cur.j = static_cast<int>((t0 - cur.P) % cur.nt);

  // Loads tile `c` into stage s (one thread).
  // Paged cache: a tile of TK keys is TK / rows page pieces (rows = min(page
  // size, TK)); lane i < NSUB handles piece i. Its physical page is looked up
  // one tile period before the copy is issued (see `ahead_pg`).
  const int pg_rows = a.block_table != nullptr ? min(a.page_size, C::TK) : C::TK;
  const int nsub = C::TK / pg_rows;
  auto lookup_page = [&](const TileCursor& c) -> int {  // this lane's piece of tile c
    if (a.block_table == nullptr || lane >= nsub) return 0;
    const int last_lp = (dec_len(a, c.b) - 1) / a.page_size;  // pages past the length are not read
    return dec_page(a, c.b, min((c.j * C::TK + lane * pg_rows) / a.page_size, last_lp));
  };
  // Loads tile c into stage s (warp-collective: lane 0 arms the barrier, the
  // lanes of the page pieces issue their copies).
  // Contiguous cache: the last tile of a unit is fetched only as far as the
  // length needs, in 16-row boxes (lane i copies rows [16 i, 16 i + 16)); the
  // rows past the length are masked (K) and zeroed (V) before use, whatever
  // the stage held.
  auto issue = [&](const TileCursor& c, int pg, int s) {
    uint8_t* kdst = ring + s * C::STAGE_BYTES;
    uint8_t* vdst = kdst + C::TILE_BYTES;
    const int hkv = c.r / a.qgroups;
    int rows16 = C::TK;  // rows copied
    if (a.block_table == nullptr) rows16 = min(C::TK, (dec_len(a, c.b) - c.j * C::TK + 15) & ~15);
    if (lane == 0) mbar_arrive_expect_tx(full + s, rows16 == C::TK ? C::STAGE_BYTES : 2 * C::KBLK * rows16 * 128);
    __syncwarp();
    if (a.block_table == nullptr) {
      const int plane = c.b * a.Hkv + hkv;
      if (rows16 == C::TK) {
        if (lane == 0) {
#pragma unroll
          for (int kb = 0; kb < C::KBLK; ++kb) {
            tma_load_3d(kdst + kb * C::BOX_BYTES, &tm_k, full + s, kb * 64, c.j * C::TK, plane);
            tma_load_3d(vdst + kb * C::BOX_BYTES, &tm_v, full + s, kb * 64, c.j * C::TK, plane);
          }
        }
      } else if (lane < rows16 / 16) {
#pragma unroll
        for (int kb = 0; kb < C::KBLK; ++kb) {
          tma_load_3d(kdst + kb * C::BOX_BYTES + lane * 16 * 128, &tm_k16, full + s, kb * 64, c.j * C::TK + 16 * lane,
                      plane);
          tma_load_3d(vdst + kb * C::BOX_BYTES + lane * 16 * 128, &tm_v16, full + s, kb * 64, c.j * C::TK + 16 * lane,
                      plane);
        }
      }
    } else if (lane < nsub) {
      const int plane = pg * a.Hkv + hkv;
      const int row = (c.j * C::TK + lane * pg_rows) % a.page_size;
#pragma unroll
      for (int kb = 0; kb < C::KBLK; ++kb) {
        tma_load_3d(kdst + kb * C::BOX_BYTES + lane * pg_rows * 128, &tm_k, full + s, kb * 64, row, plane);
        tma_load_3d(vdst + kb * C::BOX_BYTES + lane * pg_rows * 128, &tm_v, full + s, kb * 64, row, plane);
      }
    }
    if (lane == 0) fills[s] += 1;
  };

  // The first STAGES tiles are issued up front by warp 0; after that, the last
  // warp to release a stage refills it with the tile STAGES further on (`ahead`).
  TileCursor ahead = cur;
  for (int k = 0; k < C::STAGES && k < n_tiles; ++k) {
    if (warp == 0) {
      if (k == 0 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_k16);
        tma_prefetch_desc(&tm_v16);
      }
      issue(ahead, lookup_page(ahead), k);
    }
    if (k + 1 < n_tiles) dec_advance<C::TK>(a, UPB, ahead);
  }
  int ahead_pg = (C::STAGES < n_tiles) ? lookup_page(ahead) : 0;

  // Fragment coordinates (m16n8k16): lane = 4 g + t holds query row g and
  // key / value columns 2t, 2t+1 of each 8-wide n-tile.
  const int g = lane >> 2;
  const int t4 = lane & 3;
  const bool row_live = g < GC;
  // ldmatrix row addresses: lane i feeds row (i % 8) of matrix (i / 8).
  const int lm_mat = lane >> 3;
  const int lm_row = lane & 7;
  const float sl2 = a.scale_log2;

  // Q of a unit as the A operand (rows >= GC are zero): qa[kk] = {a0, a2} of k-step kk.
  auto load_q = [&](const TileCursor& c, uint32_t (&qa)[D / 16][2]) {
    const int h0 = (c.r / a.qgroups) * a.group + (c.r % a.qgroups) * GC;
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(a.q + ((size_t)c.b * a.Hq + h0 + (row_live ? g : 0)) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = row_live ? qrow[kk * 8 + t4] : 0u;
      qa[kk][1] = row_live ? qrow[kk * 8 + 4 + t4] : 0u;
    }
  };
  uint32_t qa[D / 16][2];
  load_q(cur, qa);

  // Partial pieces of this CTA (its first and/or last), settled after the stream.
  int pend_n = 0;
  int pend_u[2], pend_pieces[2], pend_b[2], pend_h0[2];
  bool pend_early[2] = {false, false};  // ticket already taken (a first piece that was not the last)
  bool pend_last[2] = {false, false};   // thread 0: the result of that early ticket

  int it_tile = 0;  // tiles of this CTA consumed so far (ring position)
  while (it_tile < n_tiles) {
    const int jbeg = cur.j;
    const int jend = min(cur.nt, jbeg + (n_tiles - it_tile));
    const int b = cur.b;
    const int h0 = (cur.r / a.qgroups) * a.group + (cur.r % a.qgroups) * GC;
    const int L = dec_len(a, b);

    float m_run = -CUDART_INF_F;  // reference max of row g (base-2 units), shared by l and o
    float l_part = 0.f;           // this lane's share of the denominator of row g
    float o[D / 8][4];            // O rows g (c0, c1) and g + 8 (c2, c3, always 0)
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    for (int jj = jbeg; jj < jend; ++jj, ++it_tile) {
      const int s = it_tile % C::STAGES;
      bool live = !*abort_flag;
      if (live && a.stall != 0 && blockIdx.x == 0 && warp == 0 && it_tile == 0) {
        // test hook: gives up after 1 ms (nothing arrives), then takes the abort path
        mbar_wait(stall_bar, 0, a.status, kSiteDecFull, abort_flag, kStallLimitNs);
        *abort_flag = 1;
        live = false;
      }
      if (live && !mbar_wait(full + s, (it_tile / C::STAGES) & 1, a.status, kSiteDecFull, abort_flag)) {
        *abort_flag = 1;
        live = false;
      }
      if (live) {
        const uint32_t kt = smem_u32(ring + s * C::STAGE_BYTES);
        const uint32_t vt = kt + C::TILE_BYTES;
        const int row0 = warp * C::KPW;          // first tile row of this warp
        const int key0 = jj * C::TK + row0;      // its key index in the sequence
        if (a.k_new != nullptr && L - 1 >= key0 && L - 1 < key0 + C::KPW) {
          // This warp's rows hold the appended token: put its K/V into the
          // stage (whatever the cache row held when it was loaded), and have
          // the first query group of the KV head store it in the cache.
          const int hkv = cur.r / a.qgroups;
          const int r = L - 1 - jj * C::TK;
          const __nv_bfloat16* src = (lane < 16 ? a.k_new : a.v_new) + ((size_t)b * a.Hkv + hkv) * D;
          uint8_t* stile = ring + s * C::STAGE_BYTES + (lane < 16 ? 0 : C::TILE_BYTES);
          for (int c = lane & 15; c < D / 8; c += 16) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + 8 * c);
            *reinterpret_cast<uint4*>(stile + (c >> 3) * C::BOX_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = w;
            if (cur.r % a.qgroups == 0) {
              __nv_bfloat16* dst = (lane < 16 ? a.k_cache : a.v_cache) + dec_row_offset(a, b, hkv, L - 1, D);
              *reinterpret_cast<uint4*>(dst + 8 * c) = w;
            }
          }
          fence_proxy_async_smem();  // before a later TMA refill overwrites the stage
          __syncwarp();
        }
        // ---- S = Q K^T for this warp's 16 keys: n-tile 0 = keys 0-7, 1 = keys 8-15
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int krow = row0 + (lm_mat >> 1) * 8 + lm_row;
          const uint32_t kbase = kt + krow * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int chunk = 2 * kk + (lm_mat & 1);
            uint32_t kb[4];
            ldsm_x4(kbase + (chunk >> 3) * C::BOX_BYTES + (((chunk & 7) ^ (krow & 7)) << 4), kb);
            mma_bf16_16816(sacc[0], qa[kk][0], 0u, qa[kk][1], 0u, kb[0], kb[1]);
            mma_bf16_16816(sacc[1], qa[kk][0], 0u, qa[kk][1], 0u, kb[2], kb[3]);
          }
        }
        // ---- mask, lazy running max, probabilities (row g; keys 8n + 2t + e)
        const int nvalid = L - key0;  // keys of this warp below the length
        float sv[4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            sv[2 * n + e] = (8 * n + 2 * t4 + e < nvalid) ? sacc[n][e] * sl2 : -CUDART_INF_F;
        float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const bool need = mx > m_run + 8.f;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2_approx(m_run - mx) : 1.f;  // 0 while m_run is -inf
          if (need) m_run = mx;
          l_part *= alpha;
#pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            o[n][0] *= alpha;
            o[n][1] *= alpha;
          }
        }
        const float m_ref = (m_run == -CUDART_INF_F) ? 0.f : m_run;
        float p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          p[i] = ex2_approx(sv[i] - m_ref);
          l_part += p[i];
        }
        const uint32_t pa0 = pack_bf16x2(p[0], p[1]);  // keys 2t, 2t+1
        const uint32_t pa2 = pack_bf16x2(p[2], p[3]);  // keys 8+2t, 8+2t+1
        // ---- rows past the length may hold anything (even NaN): zero them so
        // that 0 * V stays 0 in the MMA. Only this warp reads its rows.
        if (nvalid < C::KPW) {
          for (int i = lane; i < C::KPW * (D / 8); i += 32) {
            const int r = i / (D / 8), c = i % (D / 8);
            if (r >= max(nvalid, 0)) {
              const int row = row0 + r;
              *reinterpret_cast<uint4*>(ring + s * C::STAGE_BYTES + C::TILE_BYTES + (c >> 3) * C::BOX_BYTES +
                                        row * 128 + (((c & 7) ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();  // before a later TMA refill overwrites these rows
          __syncwarp();
        }
        // ---- O += P V: B fragments of two 8-column n-tiles per ldmatrix
        {
          const int vrow = row0 + (lm_mat & 1) * 8 + lm_row;
          const uint32_t vbase = vt + vrow * 128;
#pragma unroll
          for (int jp = 0; jp < D / 16; ++jp) {
            const int chunk = 2 * jp + (lm_mat >> 1);
            uint32_t vb[4];
            ldsm_x4_trans(vbase + (chunk >> 3) * C::BOX_BYTES + (((chunk & 7) ^ (vrow & 7)) << 4), vb);
            mma_bf16_16816(o[2 * jp], pa0, 0u, pa2, 0u, vb[0], vb[1]);
            mma_bf16_16816(o[2 * jp + 1], pa0, 0u, pa2, 0u, vb[2], vb[3]);
          }
        }
      }
      __syncwarp();  // this warp's reads of the stage are done
      int refill = 0;
      if (lane == 0) {
        __threadfence_block();
        const int done = atomicAdd(releases + s, 1) + 1;
        // Last warp off this stage: it refills it with the tile STAGES further on.
        refill = done % C::NW == 0 && it_tile + C::STAGES < n_tiles && !*abort_flag;
        if (refill) __threadfence_block();
      }
      if (__shfl_sync(0xffffffffu, refill, 0)) issue(ahead, ahead_pg, s);
      if (it_tile + C::STAGES + 1 < n_tiles) {
        dec_advance<C::TK>(a, UPB, ahead);
        ahead_pg = lookup_page(ahead);  // ready a tile period before it is needed
      }
    }

    // ---- end of the piece. Start loading the next piece's queries first.
    const int u_idx = b * UPB + cur.r;
    const long long P_u = cur.P + (long long)cur.r * cur.nt;
    const bool whole = (jbeg == 0 && jend == cur.nt);
    const int slot = static_cast<int>(blockIdx.x - P_u / chunk);
    const int pieces = static_cast<int>((P_u + cur.nt - 1) / chunk - P_u / chunk + 1);
    if (it_tile < n_tiles) {
      cur.j = jend - 1;
      dec_advance<C::TK>(a, UPB, cur);  // the piece ended at the unit's last tile
      load_q(cur, qa);
    }
    // Each warp leaves (m, l, u) of its rows; one barrier; each thread merges
    // GC*D / THREADS output elements over the warps.
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
    if (row_live) {
      if (t4 == 0) {
        wm_sm[warp * GC + g] = m_run;
        wl_sm[warp * GC + g] = l_part;
      }
      float* sl = sl_sm + (warp * GC + g) * D + 2 * t4;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) *reinterpret_cast<float2*>(sl + 8 * n) = make_float2(o[n][0], o[n][1]);
    }
    __syncthreads();
    const bool live = !*abort_flag;
    const size_t pslot = (size_t)u_idx * a.slots + slot;
    for (int i = tid; i < GC * D; i += C::THREADS) {
      const int gi = i / D, col = i % D;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < C::NW; ++w) M = fmaxf(M, wm_sm[w * GC + gi]);
      const float mr = (M == -CUDART_INF_F) ? 0.f : M;
      float Lt = 0.f, val = 0.f;
#pragma unroll
      for (int w = 0; w < C::NW; ++w) {
        const float f = ex2_approx(wm_sm[w * GC + gi] - mr);
        Lt = fmaf(wl_sm[w * GC + gi], f, Lt);
        val = fmaf(sl_sm[(w * GC + gi) * D + col], f, val);
      }
      if (!live) continue;
      const float ov = Lt > 0.f ? val / Lt : 0.f;
      const float lse2 = Lt > 0.f ? M + log2f(Lt) : -CUDART_INF_F;  // base 2
      if (whole) {
        a.o[((size_t)b * a.Hq + h0 + gi) * D + col] = __float2bfloat16_rn(ov);
        if (a.lse != nullptr && col == 0)
          a.lse[(size_t)b * a.Hq + h0 + gi] = lse2 * 0.69314718055994531f;
      } else {
        a.part_o[pslot * GC * D + i] = ov;
        if (col == 0) a.part_lse[pslot * GC + gi] = lse2;
      }
    }
    __syncthreads();  // the slices are free again
    if (!whole) {
      pend_u[pend_n] = u_idx;
      pend_pieces[pend_n] = pieces;
      pend_b[pend_n] = b;
      pend_h0[pend_n] = h0;
      // A first piece that is not also the last: thread 0 takes its ticket now
      // (its round trip then overlaps the stream); the other pieces of that
      // unit were started by the previous CTA, so it is rarely the last to
      // arrive. The barrier above ordered every thread's partial writes before
      // the ticket, a release; when it is the last, the ticket also acquires
      // the other pieces' partials.
      pend_early[pend_n] = it_tile < n_tiles;
      if (pend_early[pend_n] && tid == 0)
        pend_last[pend_n] = live && atom_add_acq_rel_gpu(a.tickets + u_idx, 1) == pieces - 1;
      ++pend_n;
    }
  }

  // ---- settle the partial pieces: the last piece of a unit to finish merges.
  if (pend_n > 0) {
    __syncthreads();  // every thread's partial writes precede thread 0's tickets (releases)
    if (tid == 0) {
      const bool live = !*abort_flag;
      for (int k = 0; k < pend_n; ++k)
        last_flag[k] = pend_early[k] ? pend_last[k]
                                     : live && atom_add_acq_rel_gpu(a.tickets + pend_u[k], 1) == pend_pieces[k] - 1;
    }
    __syncthreads();  // a last ticket (an acquire) precedes every thread's reads of the partials
    for (int k = 0; k < pend_n; ++k) {
      if (!last_flag[k]) continue;
      const int pieces = pend_pieces[k];
      const float* plse = a.part_lse + (size_t)pend_u[k] * a.slots * GC;
      const float* po = a.part_o + (size_t)pend_u[k] * a.slots * GC * D;
      for (int i = tid; i < GC * D; i += C::THREADS) {
        const int gi = i / D;
        // Up to 4 partials are loaded together (independent loads), more in a loop.
        float ls[4], os[4];
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
          ls[sp] = sp < pieces ? __ldcg(plse + sp * GC + gi) : -CUDART_INF_F;
          os[sp] = sp < pieces ? __ldcg(po + (size_t)sp * GC * D + i) : 0.f;
        }
        float mx = fmaxf(fmaxf(ls[0], ls[1]), fmaxf(ls[2], ls[3]));
        for (int sp = 4; sp < pieces; ++sp) mx = fmaxf(mx, __ldcg(plse + sp * GC + gi));
        const float mr = (mx == -CUDART_INF_F) ? 0.f : mx;
        float tot = 0.f, u = 0.f;
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
          const float wgt = ex2_approx(ls[sp] - mr);
          tot += wgt;
          u = fmaf(wgt, os[sp], u);
        }
        for (int sp = 4; sp < pieces; ++sp) {
          const float wgt = ex2_approx(__ldcg(plse + sp * GC + gi) - mr);
          tot += wgt;
          u = fmaf(wgt, __ldcg(po + (size_t)sp * GC * D + i), u);
        }
        a.o[((size_t)pend_b[k] * a.Hq + pend_h0[k] + gi) * D + (i % D)] =
            __float2bfloat16_rn(tot > 0.f ? u / tot : 0.f);
        if (a.lse != nullptr && (i % D) == 0)
          a.lse[(size_t)pend_b[k] * a.Hq + pend_h0[k] + gi] =
              tot > 0.f ? (mx + log2f(tot)) * 0.69314718055994531f : -CUDART_INF_F;
      }
      if (tid == 0) a.tickets[pend_u[k]] = 0;  // ready for the next call
    }
  }

  // Copies still in flight (only after a wait gave up) land before the CTA exits.
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    for (int s = 0; s < C::STAGES; ++s)
      if (fills[s] > 0) mbar_wait(full + s, (fills[s] - 1) & 1, a.status, kSiteDecDrain);
  }
}

}  // namespace attn_dev
